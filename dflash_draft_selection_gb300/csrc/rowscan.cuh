// rowscan.cuh -- one-pass streaming reduction of full-vocabulary logit rows.
//
// Both logit streams of the DFlash 2 path (the drafter's block logits for the
// top-16 candidates and U, the target's verify logits for p) are reductions
// of whole vocabulary rows: a running max / sum of exponentials, an argmax,
// or the best N keys.
//
// Work split.  The rows are cut into 8 KB chunks and the flat chunk sequence
// (row-major) is split into one contiguous range per CTA, equal to within a
// chunk, so every CTA streams the same number of bytes whatever the row count.
// A row that straddles two or more ranges is reduced by each of its CTAs; each
// writes a partial result to the workspace and the CTA that completes the row
// (a per-row ticket) combines the parts in CTA order and finishes the row.
// When the rows alone nearly fill the CTA slots, each CTA takes one whole row
// instead and no row is split.
//
// Streaming.  Chunk j of a CTA's range belongs to streaming warp j mod 4.
// Each streaming warp streams its chunks through a private 2-stage
// shared-memory ring filled by 1-D bulk copies (cp.async.bulk) that complete
// on per-stage mbarriers.  A warp copies an arrived chunk into registers and
// refills the stage at once, so two of its chunks are always in flight.  The
// copies read with an L2 evict-first policy: the logits are read once.
//
// Per chunk, each lane takes the maximum of its 128 (bf16) elements with
// packed bf16x2 maxima and (for the log normaliser) its sum of 2^((x-m)c)
// with packed f32x2 multiply-adds and adds.  Argmax: only lanes whose maximum
// beats the warp's best value revisit their elements.  Best N elements: a
// lane slice (the chunk's 128 elements one lane holds) whose maximum reaches
// the row's value floor is pushed as one key (its maximum, its first element)
// to the warp's ring in shared memory.  While the row streams, the CTA's
// completion warp drains the four rings into the row's sorted list of best
// slice keys and publishes the value of its N-th key as the floor.  At least N
// elements reach the floor, the best of that value and the N-th largest of the
// maxima of disjoint halves of the lane slices of the warps' first chunks of
// the row (taken together behind a named barrier).  The N best elements of
// the row then lie in the slices whose maximum reaches the N-th largest slice
// maximum F, and are ranked exactly from those slices alone, re-read once at
// the end of the row.
//
// Row ends.  The streaming warps hand each row's partial results (sums,
// argmax keys, their ring position) to the completion warp through
// double-buffered shared slots and stream on; the completion warp finishes
// the row's rings, joins the CTAs of a split row, ranks the row's elements
// and writes the outputs, and clears the row's shared state before it frees
// the slot.
//
// Waits are bounded: a warp that times out raises the error word, stops
// issuing copies, waits a bounded time for those in flight and flags its rows.
#pragma once

#include "common.cuh"

namespace dfl {

constexpr int CHUNK_BYTES = 8192;
constexpr int WSTAGES = 2;
constexpr int SCAN_WARPS = 4;
constexpr int SCAN_THREADS = SCAN_WARPS * 32 + 32;  // + one completion warp
constexpr int VEC_PER_CHUNK = CHUNK_BYTES / 16;
constexpr int VEC_PER_LANE = VEC_PER_CHUNK / 32;
constexpr int RING = 128;             // slice-key ring of a streaming warp (a power of two)
constexpr int GCAP = 256;             // element keys the completion warp gathers at once (its scratch)
constexpr int MAX_SCAN_GRID = 1024;   // CTAs of a scan launch (partial records are sized for it)
constexpr long long WAIT_CYCLES = 4000000000ll;  // ~2 s at 2 GHz
constexpr long long DRAIN_CYCLES = 200000000ll;  // ~0.1 s

struct ScanGeom {
    const char *base;  // logits
    int64_t ld_bytes;  // row stride in bytes
    int64_t V;
    int64_t rows;
    int cpr;              // chunks per row
    uint32_t last_bytes;  // bulk-copied bytes of the row's last chunk (a multiple of 16)
    int64_t total;        // rows * cpr
    const dflash2_sampling *params;
    int64_t rows_per_param;
    int64_t V_params;  // vocabulary size the sampling parameters refer to (the whole row's, for a shard)
    // Test hook (dflash2_test_hold): NULL, or a device word that every
    // streaming warp waits on, for at most hold_cycles, before its first copy.
    const unsigned int *hold;
    long long hold_cycles;
};

// The hook's current setting, process-wide (host side; set by dflash2_test_hold).
void scan_hold(const unsigned int **flag, long long *cycles);

// Partial result of a row reduced by several CTAs.
struct PartRec {
    float m, s;     // log normaliser part
    int32_t bad;
    int32_t pad;
    uint64_t keys[DFLASH2_MAX_TOPK];  // best keys, descending (keys[0] = best for an argmax)
};

// A scan's workspace: one ticket per row, one wide mark per row (the CTA,
// plus one, that left the row to its epilogue), the partial records of
// split rows.  Tickets and marks are zero between calls.
struct ScanWs {
    int32_t *tickets;  // [rows]
    int32_t *marks;    // [rows]
    PartRec *parts;    // [2 * MAX_SCAN_GRID]
};

constexpr size_t scan_ws_rows_bytes(int64_t rows) {
    return (static_cast<size_t>(rows) * sizeof(int32_t) + 255) / 256 * 256;
}
constexpr size_t scan_ws_bytes(int64_t rows) {
    return 2 * scan_ws_rows_bytes(rows) + static_cast<size_t>(2 * MAX_SCAN_GRID) * sizeof(PartRec);
}
inline ScanWs scan_ws_at(void *p, int64_t rows) {
    char *c = static_cast<char *>(p);
    ScanWs w;
    w.tickets = reinterpret_cast<int32_t *>(c);
    w.marks = reinterpret_cast<int32_t *>(c + scan_ws_rows_bytes(rows));
    w.parts = reinterpret_cast<PartRec *>(c + 2 * scan_ws_rows_bytes(rows));
    return w;
}

inline ScanGeom make_geom(const void *logits, int64_t ld, int es, int64_t V, int64_t rows,
                          const dflash2_sampling *params, int64_t rows_per_param) {
    ScanGeom g;
    g.base = static_cast<const char *>(logits);
    g.ld_bytes = ld * es;
    g.V = V;
    g.rows = rows;
    g.cpr = static_cast<int>((V * es + CHUNK_BYTES - 1) / CHUNK_BYTES);
    g.last_bytes = static_cast<uint32_t>(((V * es) - static_cast<int64_t>(g.cpr - 1) * CHUNK_BYTES) &
                                         ~static_cast<int64_t>(15));
    g.total = rows * g.cpr;
    g.params = params;
    g.rows_per_param = rows_per_param;
    g.V_params = V;
    scan_hold(&g.hold, &g.hold_cycles);
    return g;
}

// CTA b owns the flat chunks [range_begin(b), range_begin(b + 1)).
__device__ __forceinline__ int64_t range_begin(const ScanGeom &g, int64_t b) {
    return b * g.total / static_cast<int64_t>(gridDim.x);
}
// The CTA whose range holds flat chunk f: the largest b with range_begin(b) <= f.
__device__ __forceinline__ int64_t range_owner(const ScanGeom &g, int64_t f) {
    return ((f + 1) * static_cast<int64_t>(gridDim.x) + g.total - 1) / g.total - 1;
}

struct ScanSmem {
    uint64_t full[SCAN_WARPS][WSTAGES];
    uint64_t slot_full[2], slot_empty[2];  // row hand-off (count SCAN_WARPS / 1)
    unsigned int floor_ord[2];             // CTA-wide value floor of a row (ordered bits), by row parity
    unsigned int ring_head[SCAN_WARPS];    // keys pushed to each warp's ring so far
    unsigned int ring_tail[SCAN_WARPS];    // keys of each ring the completion warp has taken
    int ngather;                           // keys the completion warp has gathered into its scratch
    int nwide;                             // rows the completion warp left to the epilogue
    uint32_t lmax[2][SCAN_WARPS][DFLASH2_MAX_TOPK];  // sorted half-slice maxima of each warp's first chunk of a row
    uint64_t ring[SCAN_WARPS][RING];       // slice keys, position = count mod RING
    // Row results handed from the streaming warps to the completion warp.
    struct Hand {
        uint64_t wbest[SCAN_WARPS];
        float wm[SCAN_WARPS], wsum[SCAN_WARPS];
        int bad[SCAN_WARPS];
        unsigned int ring_end[SCAN_WARPS];  // 1 + the warp's ring count at its end of the row; 0 before
    } hand[2];
    alignas(16) unsigned char scratch[GCAP * 8];  // the completion warp's gathered keys; verify's draws
    alignas(128) unsigned char buf[SCAN_WARPS][WSTAGES][CHUNK_BYTES];
};

constexpr size_t scan_smem_bytes() { return sizeof(ScanSmem) + 128; }
// Three CTAs per SM: 228 KB of shared memory, 1 KB of it reserved per CTA.
static_assert(3 * (scan_smem_bytes() + 1024) <= 228 * 1024, "three scan CTAs must fit on an SM");

template <int R>
struct RowResult {
    WarpList<R> list;  // merged best keys (modes TOPN*)
    uint64_t best;     // best key (MODE_ARGMAX)
    float m, s;        // max and sum of 2^((x - m) c) (MODE_TOPN_LSE)
    bool bad;          // NaN seen or a wait failed
};

// ------------------------------------------------------ per-warp streams ----
// Warp w owns the chunks begin + w, begin + w + SCAN_WARPS, ... of its CTA's
// range: n_w of them.  The issue side runs WSTAGES chunks ahead of the consume side,
// across rows; both walk their position with 32-bit counters (a CTA's range
// holds far fewer than 2^31 chunks: a device buffer holds fewer than 2^27).
struct WarpStream {
    const char *iss_row;  // row of the next issue
    int iss_c;            // chunk (within its row) of the next issue
    int iss_k;            // chunks issued
    int cons_c;           // chunk (within its row) of the next consume
    int cons_r;           // row of the next consume, relative to the CTA's first row
    int cons_k;           // chunks consumed
    int n_w;              // chunks of this warp in the CTA's range
    uint32_t head;        // keys pushed to the warp's ring
    uint64_t pol;         // L2 policy of the stream: read once, evicted first
    bool aborted;
};

__device__ __forceinline__ uint32_t chunk_bulk_bytes(const ScanGeom &g, int c) {
    return c == g.cpr - 1 ? g.last_bytes : static_cast<uint32_t>(CHUNK_BYTES);
}

// Issue the warp's next chunk (lane 0) and advance the issue position.
__device__ __forceinline__ void stream_issue(ScanSmem &sm, const ScanGeom &g, WarpStream &ws, int w, int lane) {
    const int stage = ws.iss_k % WSTAGES;
    if (lane == 0) {
        const uint32_t bytes = chunk_bulk_bytes(g, ws.iss_c);
        uint64_t *bar = &sm.full[w][stage];
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, bytes);
        if (bytes)
            bulk_g2s_hint(sm.buf[w][stage], ws.iss_row + static_cast<int64_t>(ws.iss_c) * CHUNK_BYTES, bytes, bar,
                          ws.pol);
    }
    __syncwarp();
    ++ws.iss_k;
    ws.iss_c += SCAN_WARPS;
    while (ws.iss_c >= g.cpr) {
        ws.iss_c -= g.cpr;
        ws.iss_row += g.ld_bytes;
    }
}

// Test hook: lane 0 waits until *flag is nonzero, for at most max_cycles SM
// clock cycles.  True if the word was seen set.
__device__ __forceinline__ bool hold_wait(const unsigned int *flag, long long max_cycles) {
    const long long t0 = clock64();
    while (*reinterpret_cast<const volatile unsigned int *>(flag) == 0) {
        if (clock64() - t0 > max_cycles) return false;
        __nanosleep(256);
    }
    return true;
}

// Set up warp w's chunk stream over flat chunks [begin, end) and issue its
// first copies.  With the test hook set the warp first waits for the hook's
// word; if the wait runs out, the warp issues nothing, flags the error word
// and goes through its rows as after any time-out (every row bad).
__device__ __forceinline__ void stream_start(ScanSmem &sm, const ScanGeom &g, WarpStream &ws, int64_t begin,
                                             int64_t end, int w, int lane, unsigned int *err_word) {
    const int64_t len = end - begin;
    ws.n_w = len > w ? static_cast<int>((len - w + SCAN_WARPS - 1) / SCAN_WARPS) : 0;
    const int64_t f0 = begin + w;
    const int64_t r0 = f0 / g.cpr;
    ws.iss_c = ws.cons_c = static_cast<int>(f0 - r0 * g.cpr);
    ws.iss_row = g.base + r0 * g.ld_bytes;
    ws.cons_r = static_cast<int>(r0 - begin / g.cpr);
    ws.iss_k = ws.cons_k = 0;
    ws.head = 0;
    ws.pol = l2_policy_evict_first();
    ws.aborted = false;
    if (g.hold != nullptr) {
        int seen = 1;
        if (lane == 0) seen = hold_wait(g.hold, g.hold_cycles) ? 1 : 0;
        if (!__shfl_sync(FULL, seen, 0)) {
            ws.aborted = true;
            if (lane == 0) atomicOr(err_word, ERR_WAIT_TIMEOUT);
        }
    }
    for (int i = 0; i < WSTAGES && !ws.aborted && ws.iss_k < ws.n_w; ++i) stream_issue(sm, g, ws, w, lane);
}

// After a time-out: wait a bounded time for the copies still in flight.
__device__ __forceinline__ void stream_drain(ScanSmem &sm, const WarpStream &ws, int w) {
    for (int k = ws.cons_k; k < ws.iss_k; ++k)
        mbar_wait(&sm.full[w][k % WSTAGES], (k / WSTAGES) & 1, DRAIN_CYCLES);
    __syncwarp();
}

// ------------------------------------------------------------ scan state ----
// A lane slice is what one lane reads of a chunk: vectors lane + 32 q
// (q < 16) of 16 bytes, 128 bf16 or 64 f32 elements.  Its key orders slices
// by their maximum, then by the index of their first element (lower first):
// no element of the slice has a larger key.  The ragged end of a row (fewer
// than 16 bytes) enters as single elements, whose key sits just below their
// own element key; bit 31 of the low word tells them apart.
__device__ __forceinline__ uint64_t slice_key(float vmax, uint32_t base) { return make_key(vmax, base); }
__device__ __forceinline__ uint64_t tail_key(float x, uint32_t idx) { return make_key(x, idx) & ~0x80000000ull; }
__device__ __forceinline__ bool key_is_slice(uint64_t k) { return (static_cast<uint32_t>(k) & 0x80000000u) != 0; }
__device__ __forceinline__ uint32_t key_base(uint64_t k) { return ~static_cast<uint32_t>(k) & 0x7fffffffu; }

// The eight partial sums of the log normaliser (f32x2 pairs).
__device__ __forceinline__ void scale_sums(uint64_t (&acc)[4], float sc) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        acc[j] = pack2(__float_as_uint(__uint_as_float(lo32(acc[j])) * sc),
                       __float_as_uint(__uint_as_float(hi32(acc[j])) * sc));
}
__device__ __forceinline__ float sum_sums(const uint64_t (&acc)[4]) {
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) s += __uint_as_float(lo32(acc[j])) + __uint_as_float(hi32(acc[j]));
    return s;
}

template <int R>
struct ScanState {
    float bv;   // argmax: this lane's best value and its id
    int32_t bi;
    float bw;   // argmax: the warp's best value (warp-uniform)
    float m, negmc, c;
    uint64_t acc[4];  // sum of 2^((x - m) c): eight partial sums as f32x2 pairs
    float lo;          // value floor: at least N elements of the row reach it; warp-uniform
    bool bad;
};

// A chunk's 16-byte vectors as one lane holds them in registers: vector q is
// lane + 32 q; vectors past the chunk's data hold -inf.
template <bool BF16>
struct VecLoad;
template <>
struct VecLoad<true> {
    static constexpr int VE = 8;
    static constexpr uint32_t NEG_WORD = 0xff80ff80u;  // two bf16 -inf
    __device__ __forceinline__ static void unpack(uint4 w, float (&x)[8]) {
        x[0] = bf16lo(w.x);
        x[1] = bf16hi(w.x);
        x[2] = bf16lo(w.y);
        x[3] = bf16hi(w.y);
        x[4] = bf16lo(w.z);
        x[5] = bf16hi(w.z);
        x[6] = bf16lo(w.w);
        x[7] = bf16hi(w.w);
    }
    // NaN-propagating maximum of a vector.
    __device__ __forceinline__ static float vmax(uint4 w) {
        const uint32_t mm = bmax2_nan(bmax2_nan(w.x, w.y), bmax2_nan(w.z, w.w));
        return fmax_nan(bf16lo(mm), bf16hi(mm));
    }
    // NaN-propagating maxima of two disjoint halves of the lane's elements
    // (the low and the high bf16 of every word; packed bf16x2 maxima).
    __device__ __forceinline__ static void lane_max2(const uint4 (&v)[VEC_PER_LANE], float &m0, float &m1) {
        uint32_t a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = NEG_WORD;
#pragma unroll
        for (int q = 0; q < VEC_PER_LANE; ++q) {
            const int h = (q & 1) * 4;
            a[h + 0] = bmax2_nan(a[h + 0], v[q].x);
            a[h + 1] = bmax2_nan(a[h + 1], v[q].y);
            a[h + 2] = bmax2_nan(a[h + 2], v[q].z);
            a[h + 3] = bmax2_nan(a[h + 3], v[q].w);
        }
        const uint32_t mm = bmax2_nan(bmax2_nan(bmax2_nan(a[0], a[1]), bmax2_nan(a[2], a[3])),
                                      bmax2_nan(bmax2_nan(a[4], a[5]), bmax2_nan(a[6], a[7])));
        m0 = bf16lo(mm);
        m1 = bf16hi(mm);
    }
    // acc[j] += (2^(lo_j c + negmc), 2^(hi_j c + negmc)) for the bf16 pair in
    // word j of the vector (packed f32x2 arithmetic; cc, nn hold c and negmc
    // in both halves).
    __device__ __forceinline__ static void accumulate(uint4 w, uint64_t cc, uint64_t nn, uint64_t (&acc)[4]) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint64_t x = pack2(ws[j] << 16, ws[j] & 0xffff0000u);
            const uint64_t t = fma2(x, cc, nn);
            acc[j] = add2(acc[j], pack2(__float_as_uint(ex2(__uint_as_float(lo32(t)))),
                                        __float_as_uint(ex2(__uint_as_float(hi32(t))))));
        }
    }
    __device__ __forceinline__ static float scalar(const char *row, int64_t i) {
        const unsigned short b = reinterpret_cast<const unsigned short *>(row)[i];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
};
template <>
struct VecLoad<false> {
    static constexpr int VE = 4;
    static constexpr uint32_t NEG_WORD = 0xff800000u;  // f32 -inf
    __device__ __forceinline__ static void unpack(uint4 w, float (&x)[4]) {
        x[0] = __uint_as_float(w.x);
        x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z);
        x[3] = __uint_as_float(w.w);
    }
    __device__ __forceinline__ static float vmax(uint4 w) {
        return fmax_nan(fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                        fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
    // NaN-propagating maxima of two disjoint halves of the lane's vectors.
    __device__ __forceinline__ static void lane_max2(const uint4 (&v)[VEC_PER_LANE], float &m0, float &m1) {
        float a[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
        for (int q = 0; q < VEC_PER_LANE; ++q) a[q & 3] = fmax_nan(a[q & 3], vmax(v[q]));
        m0 = fmax_nan(a[0], a[1]);
        m1 = fmax_nan(a[2], a[3]);
    }
    __device__ __forceinline__ static void accumulate(uint4 w, uint64_t cc, uint64_t nn, uint64_t (&acc)[4]) {
        const uint64_t t0 = fma2(pack2(w.x, w.y), cc, nn), t1 = fma2(pack2(w.z, w.w), cc, nn);
        acc[0] = add2(acc[0], pack2(__float_as_uint(ex2(__uint_as_float(lo32(t0)))),
                                    __float_as_uint(ex2(__uint_as_float(hi32(t0))))));
        acc[1] = add2(acc[1], pack2(__float_as_uint(ex2(__uint_as_float(lo32(t1)))),
                                    __float_as_uint(ex2(__uint_as_float(hi32(t1))))));
    }
    __device__ __forceinline__ static float scalar(const char *row, int64_t i) {
        return reinterpret_cast<const float *>(row)[i];
    }
};

// Bitonic sort of one value per lane, descending across the warp.
template <typename T>
__device__ __forceinline__ T warp_sort_desc(T v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const T o = __shfl_xor_sync(FULL, v, j);
            const bool desc = (lane & k) == 0 || k == 32;
            const bool lower = (lane & j) == 0;
            const T hi = v > o ? v : o, lo = v > o ? o : v;
            v = (lower == desc) ? hi : lo;
        }
    }
    return v;
}

// Top 32 of two descending lists of 32 values (one per lane), descending.
__device__ __forceinline__ uint32_t warp_merge_desc_u32(uint32_t a, uint32_t b, int lane) {
    const uint32_t rev = __shfl_sync(FULL, b, 31 - lane);
    uint32_t v = a > rev ? a : rev;  // bitonic
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        const uint32_t o = __shfl_xor_sync(FULL, v, d);
        v = ((lane & d) == 0) ? (v > o ? v : o) : (v > o ? o : v);
    }
    return v;
}

// Named barrier 1 (even rows of a CTA) or 3 (odd rows) over the first
// `threads` threads that reach it (a multiple of 32).  Alternating the id
// keeps the barriers of consecutive rows apart: a warp starts row r + 2 only
// after the completion warp took row r, i.e. after every warp left row r's
// barrier.
__device__ __forceinline__ void row_barrier(int parity, int threads) {
    if (parity == 0)
        asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
    else
        asm volatile("bar.sync 3, %0;" ::"r"(threads) : "memory");
}

// Publish a value floor for the row to the other warps of the CTA.
__device__ __forceinline__ void publish_floor(ScanSmem &sm, int rp, float v, int lane) {
    if (lane == 0 && v > NEG_INF) atomicMax(&sm.floor_ord[rp], f2ord(v));
}

// Sort `n` keys of a buffer into the list (32 keys at a time).  Warp-uniform.
template <int R>
__device__ __forceinline__ void merge_buffer(WarpList<R> &list, const uint64_t *buf, int n, int lane) {
    for (int base = 0; base < n; base += 32) {
        const uint64_t k = base + lane < n ? buf[base + lane] : 0;
        WarpList<R> o;
        o.k[0] = warp_sort_desc(k, lane);
#pragma unroll
        for (int r = 1; r < R; ++r) o.k[r] = 0;
        list.merge(o, lane);
    }
}

// Push the keys of the lanes with `lf` to warp w's ring, waiting (bounded)
// for the completion warp to make room.  False after a time-out (or once the
// warp's stream gave up).  Warp-uniform.
__device__ __forceinline__ bool ring_push(ScanSmem &sm, WarpStream &ws, int w, int lane, bool lf, uint64_t key) {
    const uint32_t bal = __ballot_sync(FULL, lf);
    if (bal == 0) return true;
    if (ws.aborted) return false;
    const uint32_t n = __popc(bal);
    int ok = 1;
    if (lane == 0) {
        const long long t0 = clock64();
        while (ws.head + n - *reinterpret_cast<volatile unsigned int *>(&sm.ring_tail[w]) > RING) {
            if (clock64() - t0 > WAIT_CYCLES) {
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
    }
    if (!__shfl_sync(FULL, ok, 0)) return false;
    if (lf) sm.ring[w][(ws.head + __popc(bal & ((1u << lane) - 1u))) & (RING - 1)] = key;
    __syncwarp();
    ws.head += n;
    if (lane == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile unsigned int *>(&sm.ring_head[w]) = ws.head;
    }
    return true;
}

// A ring push that timed out: the row is bad and the warp's stream gives up.
__device__ __forceinline__ void push_failed(WarpStream &ws, bool &bad, int lane, unsigned int *err_word) {
    bad = true;
    if (!ws.aborted && lane == 0) atomicOr(err_word, ERR_WAIT_TIMEOUT);
    ws.aborted = true;
}

// One element of the ragged end of a row (lane 0 holds it); warp-uniform.
template <int R, int MODE>
__device__ __forceinline__ void scan_one(ScanSmem &sm, WarpStream &ws, ScanState<R> &st, float x, uint32_t idx,
                                         bool valid, int w, int lane, unsigned int *err_word) {
    if (valid && x != x) st.bad = true;
    if (MODE == MODE_ARGMAX) {
        if (valid && x > st.bv) {
            st.bv = x;
            st.bi = static_cast<int32_t>(idx);
        }
        st.bw = warp_max_f(st.bv);
        return;
    }
    if (MODE == MODE_TOPN_LSE && valid) {
        if (x > st.m) {
            scale_sums(st.acc, ex2((st.m - x) * st.c));
            st.m = x;
            st.negmc = -x * st.c;
        }
        if (st.m != NEG_INF)
            st.acc[0] = pack2(__float_as_uint(__uint_as_float(lo32(st.acc[0])) + ex2(fmaf(x, st.c, st.negmc))),
                              hi32(st.acc[0]));
    }
    const bool c = valid && x == x && x >= st.lo;
    if (!ring_push(sm, ws, w, lane, c, tail_key(x, idx))) push_failed(ws, st.bad, lane, err_word);
}

// First chunk of each warp in the row (modes TOPN*, N <= R * 32): each lane
// offers the maxima m0, m1 of two disjoint halves of its slice; at least N
// elements reach the N-th largest of them.  When several warps hold chunks
// of the row (`expect` of them, from w0 on cyclically), each publishes its
// sorted maxima, waits for the others (named barrier) and merges their lists:
// a floor from up to 4 chunks instead of one.  A warp whose chunk did not
// arrive takes part with -inf maxima, so the barrier always completes.
template <int R>
__device__ __forceinline__ void first_floor(ScanSmem &sm, float &lo, float m0, float m1, int nsel, int expect, int w0,
                                            int rp, int w, int lane) {
    const uint32_t o0 = warp_sort_desc(f2ord(m0 == m0 ? m0 : NEG_INF), lane);
    const uint32_t o1 = warp_sort_desc(f2ord(m1 == m1 ? m1 : NEG_INF), lane);
    if (R == 1) {  // 32-bit lists: the top 32 of the lane maxima
        uint32_t o = warp_merge_desc_u32(o0, o1, lane);
        if (expect > 1) {
            sm.lmax[rp][w][lane] = o;
            row_barrier(rp, expect * 32);
#pragma unroll 1
            for (int i = 0; i < expect; ++i) {
                const int u = (w0 + i) % SCAN_WARPS;
                if (u != w) o = warp_merge_desc_u32(o, sm.lmax[rp][u][lane], lane);
            }
        }
        lo = fmaxf(lo, ord2f(__shfl_sync(FULL, o, nsel - 1)));
        publish_floor(sm, rp, lo, lane);
        return;
    }
    WarpList<R> L, o;
    L.clear();
    o.clear();
    L.k[0] = static_cast<uint64_t>(o0) << 32;
    o.k[0] = static_cast<uint64_t>(o1) << 32;
    L.merge(o, lane);
    if (expect > 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) sm.lmax[rp][w][r * 32 + lane] = static_cast<uint32_t>(L.k[r] >> 32);
        row_barrier(rp, expect * 32);
#pragma unroll 1
        for (int i = 0; i < expect; ++i) {
            const int u = (w0 + i) % SCAN_WARPS;
            if (u != w) {
#pragma unroll
                for (int r = 0; r < R; ++r) o.k[r] = static_cast<uint64_t>(sm.lmax[rp][u][r * 32 + lane]) << 32;
                L.merge(o, lane);
            }
        }
    }
    lo = fmaxf(lo, ord2f(static_cast<uint32_t>(L.at(nsel - 1) >> 32)));
    publish_floor(sm, rp, lo, lane);
}

// One chunk of a row held in registers (`v`: nvt vectors of data, lane
// maximum `cmax`), first element e0.  Warp-uniform.
template <int R, int MODE, bool BF16>
__device__ __forceinline__ void consume_chunk(ScanSmem &sm, WarpStream &ws, ScanState<R> &st,
                                              const uint4 (&v)[VEC_PER_LANE], int nvt, float cmax, uint32_t e0,
                                              int w, int lane, int rp, unsigned int *err_word) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    if (cmax != cmax) st.bad = true;
    if (MODE == MODE_ARGMAX) {
        const bool f = cmax > st.bw;
        if (f) {  // rare after the first chunks: the lane's new best, in index order
            float t = st.bw;
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q) {
                if (VL::vmax(v[q]) > t) {
                    float x[VE];
                    VL::unpack(v[q], x);
#pragma unroll
                    for (int e = 0; e < VE; ++e) {
                        if (x[e] > t) {
                            t = x[e];
                            st.bv = x[e];
                            st.bi = static_cast<int32_t>(e0 + (lane + q * 32) * VE + e);
                        }
                    }
                }
            }
        }
        if (__any_sync(FULL, f)) st.bw = warp_max_f(st.bv);
        return;
    }
    if (MODE == MODE_TOPN_LSE) {
        if (cmax > st.m) {  // rare after the first chunks: rescale once per chunk
            scale_sums(st.acc, ex2((st.m - cmax) * st.c));
            st.m = cmax;
            st.negmc = -cmax * st.c;
        }
        if (st.m != NEG_INF) {
            const uint64_t cc = pack2(__float_as_uint(st.c), __float_as_uint(st.c));
            const uint64_t nn = pack2(__float_as_uint(st.negmc), __float_as_uint(st.negmc));
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q) VL::accumulate(v[q], cc, nn, st.acc);
        }
    }
    // The CTA's floor for the row (one read, broadcast).
    uint32_t so = lane == 0 ? *reinterpret_cast<volatile unsigned int *>(&sm.floor_ord[rp]) : 0u;
    so = __shfl_sync(FULL, so, 0);
    if (so != 0) st.lo = fmaxf(st.lo, ord2f(so));
    const bool lf = lane < nvt && cmax >= st.lo;  // NaN never passes
    if (!ring_push(sm, ws, w, lane, lf, slice_key(cmax, e0 + lane * VE))) push_failed(ws, st.bad, lane, err_word);
}

// A streaming warp's results for the row into hand-off slot rp; the warp's
// arrival on slot_full[rp] (count SCAN_WARPS) publishes them.  Its ring count
// goes last: once the completion warp sees it, it knows where the warp's keys
// of the row end.
template <int R>
__device__ __forceinline__ void hand_off_warp(ScanSmem &sm, const WarpStream &ws, int rp, int w, int lane,
                                              const ScanState<R> &st) {
    ScanSmem::Hand &h = sm.hand[rp];
    const uint64_t kb = warp_max_u64(st.bi >= 0 ? make_key(st.bv, static_cast<uint32_t>(st.bi)) : 0);
    float mm = st.m, s = sum_sums(st.acc);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        const float m2 = __shfl_xor_sync(FULL, mm, d);
        const float s2 = __shfl_xor_sync(FULL, s, d);
        lse_combine(mm, s, m2, s2, st.c);
    }
    const bool bad = __any_sync(FULL, st.bad);
    if (lane == 0) {
        h.wbest[w] = kb;
        h.wm[w] = mm;
        h.wsum[w] = s;
        h.bad[w] = bad ? 1 : 0;
        __threadfence_block();
        *reinterpret_cast<volatile unsigned int *>(&h.ring_end[w]) = ws.head + 1u;
        mbar_arrive(&sm.slot_full[rp]);
    }
}

// A streaming warp's part of the CTA's row `rrel` (global row `row`):
// consume the warp's chunks of it and hand the warp's partial results to the
// completion warp.  Every row of the range goes through here (rows that need
// no scan with `skip`), so that the chunk streams stay in step.  `expect`
// warps, from warp w0 on (cyclically), hold a chunk of the row.
template <int R, int MODE, bool BF16>
__device__ __forceinline__ void scan_row(ScanSmem &sm, const ScanGeom &g, WarpStream &ws, const RowTask &task,
                                         int64_t row, int rrel, int expect, int w0, bool skip,
                                         unsigned int *err_word) {
    using VL = VecLoad<BF16>;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int CE = CHUNK_BYTES / esz;
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int nsel = task.nsel;
    const int rp = rrel & 1;

    // Slot rp (hand-off, floor) is free once row rrel - 2 was taken.
    bool slot_ok = true;
    if (rrel >= 2) slot_ok = __all_sync(FULL, mbar_wait(&sm.slot_empty[rp], ((rrel >> 1) - 1) & 1, WAIT_CYCLES));
    if (!slot_ok && lane == 0) atomicOr(err_word, ERR_WAIT_TIMEOUT);

    ScanState<R> st;
    st.bv = NEG_INF;
    st.bi = -1;
    st.bw = NEG_INF;
    st.m = NEG_INF;
#pragma unroll
    for (int j = 0; j < 4; ++j) st.acc[j] = 0;
    st.negmc = 0.0f;
    st.c = LOG2E / task.T;
    st.bad = !slot_ok;
    st.lo = NEG_INF;

    bool first = true;
    while (ws.cons_k < ws.n_w && ws.cons_r == rrel) {
        const int stage = ws.cons_k % WSTAGES;
        bool ok = !ws.aborted && mbar_wait(&sm.full[w][stage], (ws.cons_k / WSTAGES) & 1, WAIT_CYCLES);
        ok = __all_sync(FULL, ok);
        if (!ok && !ws.aborted) {
            ws.aborted = true;
            if (lane == 0) atomicOr(err_word, ERR_WAIT_TIMEOUT);
        }
        if (!ok) st.bad = true;
        const int c = ws.cons_c;
        const int bulk = static_cast<int>(chunk_bulk_bytes(g, c));
        const int nvt = bulk >> 4;  // vectors in the chunk
        const bool compute = ok && !skip;
        // Copy the lane's vectors into registers, then refill the stage.
        uint4 v[VEC_PER_LANE];
        const unsigned char *tile = sm.buf[w][stage];
        if (compute && nvt == VEC_PER_CHUNK) {  // every chunk but a row's last
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q) v[q] = *reinterpret_cast<const uint4 *>(tile + (lane + q * 32) * 16);
        } else {
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q) {
                const int vi = lane + q * 32;
                v[q] = (compute && vi < nvt) ? *reinterpret_cast<const uint4 *>(tile + vi * 16)
                                             : make_uint4(VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD);
            }
        }
        __syncwarp();
        if (ok) {
            ++ws.cons_k;
            if (ws.iss_k < ws.n_w) stream_issue(sm, g, ws, w, lane);
        }
        float m0 = NEG_INF, m1 = NEG_INF;
        if (compute) VL::lane_max2(v, m0, m1);
        const float cmax = fmax_nan(m0, m1);
        if (MODE != MODE_ARGMAX && first && !skip)
            first_floor<R>(sm, st.lo, m0, m1, nsel, expect, w0, rp, w, lane);
        if (compute) {
            const uint32_t e0 = static_cast<uint32_t>(c) * CE;
            consume_chunk<R, MODE, BF16>(sm, ws, st, v, nvt, cmax, e0, w, lane, rp, err_word);
            // Ragged end of the row (fewer than 16 bytes), read by lane 0.
            if (c == g.cpr - 1) {
                const char *rbase = g.base + row * g.ld_bytes;
                const int64_t cnt = g.V - e0;
                for (int64_t i = e0 + bulk / esz; i < e0 + cnt; ++i) {
                    const float xi = lane == 0 ? VL::scalar(rbase, i) : NEG_INF;
                    scan_one<R, MODE>(sm, ws, st, xi, static_cast<uint32_t>(i), lane == 0, w, lane, err_word);
                }
            }
        }
        first = false;
        // After a time-out nothing more is issued or waited for (cons_k stays
        // behind iss_k for the drain); the position still advances.
        ws.cons_c += SCAN_WARPS;
        while (ws.cons_c >= g.cpr) {
            ws.cons_c -= g.cpr;
            ++ws.cons_r;
        }
    }

    hand_off_warp(sm, ws, rp, w, lane, st);
}

// Offer every element that reaches `F` of the lane slice starting at element
// `base` (or, with !slice, the single element `base` of value `x1`) to the
// element list `out`, for the lanes with `take`, one element per lane at a
// time; `otau` is out's N-th key.  A slice is visited in groups of vectors of
// 64 elements.  Warp-uniform.
template <int R, bool BF16>
__device__ __forceinline__ void offer_slices(const ScanGeom &g, const char *rowp, bool take, uint32_t base, bool slice,
                                             float x1, float F, int nsel, int lane, WarpList<R> &out, uint64_t &otau) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int CE = CHUNK_BYTES / esz;
    constexpr int GV = 64 / VE;                 // vectors per group
    constexpr int NG = VEC_PER_LANE / GV;       // groups per slice
    static_assert(NG * GV == VEC_PER_LANE, "slices split into whole groups");
    int lin = 0, bulk = 0;
    if (slice) {
        const int c = static_cast<int>(base / CE);
        lin = static_cast<int>((base % CE) / VE);
        bulk = static_cast<int>(chunk_bulk_bytes(g, c));
    }
#pragma unroll 1
    for (int gi = 0; gi < NG; ++gi) {
        uint64_t cm = 0;
        if (take) {
            if (slice) {
#pragma unroll
                for (int j = 0; j < GV; ++j) {
                    const int q = gi * GV + j;
                    if ((lin + q * 32) * 16 < bulk) {
                        const uint4 v = __ldcg(
                            reinterpret_cast<const uint4 *>(rowp + static_cast<int64_t>(base + q * 32 * VE) * esz));
                        float x[VE];
                        VL::unpack(v, x);
#pragma unroll
                        for (int e = 0; e < VE; ++e)
                            if (x[e] >= F) cm |= 1ull << (j * VE + e);  // NaN never passes
                    }
                }
            } else if (gi == 0) {
                cm = 1;
            }
        }
        while (__any_sync(FULL, cm != 0)) {
            uint64_t key = 0;
            if (cm) {
                const int b = __ffsll(static_cast<long long>(cm)) - 1;
                cm &= cm - 1;
                if (slice) {
                    const uint32_t idx = base + (gi * GV + b / VE) * 32 * VE + (b % VE);
                    key = make_key(VL::scalar(rowp, idx), idx);
                } else {
                    key = make_key(x1, base);
                }
                if (key <= otau) key = 0;
            }
            if (__any_sync(FULL, key != 0)) {
                WarpList<R> o;
                o.k[0] = warp_sort_desc(key, lane);
#pragma unroll
                for (int r = 1; r < R; ++r) o.k[r] = 0;
                out.merge(o, lane);
                otau = out.at(nsel - 1);
            }
        }
    }
}

// Completion warp: merge the batch's ring keys (one per lane, 0 for none)
// whose value reaches the row's floor F into the row's list of best slice
// keys (N-th key `tau`), then publish the list's N-th value as the floor.
// Keys tied with F stay: the elements of tied slices are ranked by index.
// Warp-uniform.
template <int R>
__device__ __forceinline__ void merge_ring_keys(ScanSmem &sm, uint64_t k, int rp, int nsel, WarpList<R> &list,
                                                uint64_t &tau, int lane) {
    uint32_t so = lane == 0 ? *reinterpret_cast<volatile unsigned int *>(&sm.floor_ord[rp]) : 0u;
    so = __shfl_sync(FULL, so, 0);
    float F = so != 0 ? ord2f(so) : NEG_INF;
    if (tau != 0) F = fmaxf(F, key_val(tau));
    const bool take = k != 0 && key_val(k) >= F;
    if (!__any_sync(FULL, take)) return;
    WarpList<R> o;
    o.k[0] = warp_sort_desc(take ? k : 0ull, lane);
#pragma unroll
    for (int r = 1; r < R; ++r) o.k[r] = 0;
    list.merge(o, lane);
    const uint64_t t = list.at(nsel - 1);
    if (t > tau) {
        tau = t;
        publish_floor(sm, rp, key_val(t), lane);
    }
}

// Completion warp (modes TOPN*): the best slice keys of the CTA's part of
// the row in slot rp.  Drains the four rings (taken positions `tail`, kept
// across rows) while the streaming warps push to them, 32 keys a batch, until
// every warp has handed the row off and its keys of the row are taken.  While
// the rings are empty it sleeps on the slot's hand-off barrier (phase
// `parity`), which wakes it as soon as the last warp hands off.  False after
// a time-out with nothing to take.
template <int R>
__device__ __forceinline__ bool refine_row(ScanSmem &sm, int rp, uint32_t parity, int nsel,
                                           uint32_t (&tail)[SCAN_WARPS], WarpList<R> &list, int lane) {
    list.clear();
    uint64_t tau = 0;
    long long t0 = clock64();
    unsigned int nap = 128;  // ns; doubles while the rings stay empty (the hand-off wakes the warp)
    while (true) {
        // Lane w < 4 reads ring w's count, then its row-end mark: a warp that
        // has left the row wrote its mark before pushing keys of the next.
        uint32_t hv = 0, rv = 0;
        if (lane < SCAN_WARPS) hv = *reinterpret_cast<volatile unsigned int *>(&sm.ring_head[lane]);
        __threadfence_block();
        if (lane < SCAN_WARPS) rv = *reinterpret_cast<volatile unsigned int *>(&sm.hand[rp].ring_end[lane]);
        __syncwarp();  // the keys below are read by other lanes than the counts
        uint64_t k = 0;
        int nb = 0;
        bool finished = true;
#pragma unroll
        for (int w = 0; w < SCAN_WARPS; ++w) {
            const uint32_t head = __shfl_sync(FULL, hv, w);
            const uint32_t re = __shfl_sync(FULL, rv, w);
            const uint32_t lim = re != 0 ? re - 1u : head;
            const uint32_t avail = lim - tail[w];
            const uint32_t room = static_cast<uint32_t>(32 - nb);
            const uint32_t n = avail < room ? avail : room;
            if (lane >= nb && lane < nb + static_cast<int>(n)) k = sm.ring[w][(tail[w] + (lane - nb)) & (RING - 1)];
            tail[w] += n;
            nb += static_cast<int>(n);
            if (re == 0 || n < avail) finished = false;
        }
        if (nb > 0) {
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
#pragma unroll
                for (int w = 0; w < SCAN_WARPS; ++w)
                    *reinterpret_cast<volatile unsigned int *>(&sm.ring_tail[w]) = tail[w];
            }
            merge_ring_keys<R>(sm, k, rp, nsel, list, tau, lane);
            t0 = clock64();
            nap = 128;
        } else if (finished) {
            return true;
        } else {
            if (clock64() - t0 > WAIT_CYCLES) return false;
            mbar_try_wait_ns(&sm.slot_full[rp], parity, nap);
            if (nap < 1600) nap *= 2;
        }
    }
}

// Completion warp: the CTA's result for its row rrel.  Modes TOPN* first
// collect the row's best slice keys from the rings; then a bounded wait for
// the streaming warps' hand-offs (a time-out marks the row bad and stops
// further waits), merged over the warps; then clear the row's shared state
// and free the slot.
template <int R, int MODE, bool BF16>
__device__ __forceinline__ void take_row(ScanSmem &sm, const ScanGeom &g, int64_t row, RowResult<R> &res, int rrel,
                                         float c, int nsel, uint32_t (&tail)[SCAN_WARPS], bool &aborted, int lane,
                                         unsigned int *err_word) {
    const int rp = rrel & 1;
    res.list.clear();
    res.best = 0;
    res.m = NEG_INF;
    res.s = 0.0f;
    bool ok = !aborted;
    if (MODE != MODE_ARGMAX && ok) ok = refine_row<R>(sm, rp, (rrel >> 1) & 1, nsel, tail, res.list, lane);
    ok = ok && mbar_wait(&sm.slot_full[rp], (rrel >> 1) & 1, WAIT_CYCLES);
    ok = __all_sync(FULL, ok);
    if (!ok && !aborted && lane == 0) atomicOr(err_word, ERR_WAIT_TIMEOUT);
    if (!ok) aborted = true;
    const ScanSmem::Hand &h = sm.hand[rp];
    res.bad = !ok;
    if (ok) {
        for (int u = 0; u < SCAN_WARPS; ++u) {
            res.bad |= h.bad[u] != 0;
            if (MODE == MODE_ARGMAX) res.best = h.wbest[u] > res.best ? h.wbest[u] : res.best;
            if (MODE == MODE_TOPN_LSE) lse_combine(res.m, res.s, h.wm[u], h.wsum[u], c);
        }
    }
    __syncwarp();
    if (lane == 0) {
        sm.floor_ord[rp] = 0;
#pragma unroll
        for (int u = 0; u < SCAN_WARPS; ++u) sm.hand[rp].ring_end[u] = 0;
        mbar_arrive(&sm.slot_empty[rp]);
    }
}

// Completion warp, once per row (modes TOPN*): the N best elements of the row
// from its best slice keys L.  F, the N-th largest slice maximum, is reached
// by at least N elements, so every one of the N best elements lies in a slice
// whose maximum reaches F: re-read those slices (all loads of a list register
// in flight at once), gather their elements that reach F in shared memory
// (cursor `ngather`) and rank them.  If the list is full with its last key
// tied at F (slices tied at F may have been left out), or the gathered
// elements overflow the buffer, rank every slice of the row instead.
// Returns element keys.
template <int R, bool BF16>
__device__ __forceinline__ WarpList<R> extract_topn(const ScanGeom &g, int64_t row, const WarpList<R> &L, int nsel,
                                                    unsigned char *scratch, int *ngather, int lane) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int CE = CHUNK_BYTES / esz;
    const char *rowp = g.base + row * g.ld_bytes;
    const uint64_t kN = L.at(nsel - 1);
    const float F = kN ? key_val(kN) : NEG_INF;
    const uint64_t kL = L.at(R * 32 - 1);
    WarpList<R> out;
    out.clear();
    uint64_t otau = 0;
    uint64_t *gbuf = reinterpret_cast<uint64_t *>(scratch);
    if (!(kL != 0 && key_val(kL) == F)) {
        // Lane p holds list entry p (p = r*32 + lane): it loads its slice
        // (all loads in flight at once), marks the vectors whose maximum
        // reaches F and appends their elements that reach F (or its single
        // tail element) to the scratch through a shared cursor; the sort
        // below makes their order irrelevant.  The per-element work runs in
        // a rolled loop: this code runs once per row, cold, and stays small.
        if (lane == 0) *ngather = 0;
        __syncwarp();
#pragma unroll 1
        for (int r = 0; r < R; ++r) {
            uint64_t k = L.k[0];
#pragma unroll
            for (int rr = 1; rr < R; ++rr)
                if (rr == r) k = L.k[rr];
            const bool take = k != 0 && key_val(k) >= F;
            const uint32_t base = key_base(k);
            const bool slice = key_is_slice(k);
            int lin = 0, nvt = 0;
            if (slice) {
                const int c = static_cast<int>(base / CE);
                lin = static_cast<int>((base % CE) / VE);
                nvt = static_cast<int>(chunk_bulk_bytes(g, c)) >> 4;
            }
            uint4 v[VEC_PER_LANE];
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q) {
                v[q] = make_uint4(VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD);
                if (take && slice && lin + q * 32 < nvt)
                    v[q] = __ldcg(reinterpret_cast<const uint4 *>(rowp + static_cast<int64_t>(base + q * 32 * VE) * esz));
            }
            uint32_t qm = 0;
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q)
                if (take && slice && lin + q * 32 < nvt && VL::vmax(v[q]) >= F) qm |= 1u << q;  // NaN never passes
            if (take && !slice) {
                const int pos = atomicAdd(ngather, 1);
                if (pos < GCAP) gbuf[pos] = make_key(key_val(k), base);
            }
#pragma unroll 1
            while (qm) {
                const int q = __ffs(qm) - 1;
                qm &= qm - 1;
                uint4 u = v[0];
#pragma unroll
                for (int j = 1; j < VEC_PER_LANE; ++j)
                    if (j == q) u = v[j];
                float x[VE];
                VL::unpack(u, x);
                const uint32_t i0 = base + static_cast<uint32_t>(q * 32 * VE);
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                    if (x[e] >= F) {
                        const int pos = atomicAdd(ngather, 1);
                        if (pos < GCAP) gbuf[pos] = make_key(x[e], i0 + e);
                    }
                }
            }
        }
        __syncwarp();
        // one read, broadcast: every lane takes the same branch, and all have
        // read the cursor before lane 0 resets it below
        const int total = __shfl_sync(FULL, *reinterpret_cast<volatile int *>(ngather), 0);
        if (total <= GCAP) {
            merge_buffer<R>(out, gbuf, total, lane);
            return out;
        }
    }
    // A slice tied at F may have been left out of the list (always possible
    // when the list is exactly N long), or the listed slices held more than
    // the scratch: gather every element of the row that reaches F, in one
    // pass (a vector whose maximum falls below F adds nothing).
    if (lane == 0) *ngather = 0;
    __syncwarp();
#pragma unroll 1
    for (int c = 0; c < g.cpr; ++c) {
        const int nvt = static_cast<int>(chunk_bulk_bytes(g, c)) >> 4;
        const uint32_t cb = static_cast<uint32_t>(c) * CE;
        const uint4 *cp = reinterpret_cast<const uint4 *>(rowp + static_cast<int64_t>(cb) * esz);
        uint4 v[VEC_PER_LANE];
#pragma unroll
        for (int q = 0; q < VEC_PER_LANE; ++q)
            v[q] = q * 32 + lane < nvt ? __ldcs(cp + q * 32 + lane)
                                       : make_uint4(VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD);
        uint32_t qm = 0;
#pragma unroll
        for (int q = 0; q < VEC_PER_LANE; ++q)
            if (q * 32 + lane < nvt && VL::vmax(v[q]) >= F) qm |= 1u << q;
#pragma unroll 1
        while (qm) {
            const int q = __ffs(qm) - 1;
            qm &= qm - 1;
            uint4 u = v[0];
#pragma unroll
            for (int j = 1; j < VEC_PER_LANE; ++j)
                if (j == q) u = v[j];
            float x[VE];
            VL::unpack(u, x);
            const uint32_t i0 = cb + static_cast<uint32_t>((q * 32 + lane) * VE);
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                if (x[e] >= F) {
                    const int pos = atomicAdd(ngather, 1);
                    if (pos < GCAP) gbuf[pos] = make_key(x[e], i0 + e);
                }
            }
        }
    }
    {
        const int64_t t0 = static_cast<int64_t>(g.cpr - 1) * CE + chunk_bulk_bytes(g, g.cpr - 1) / esz;
        for (int64_t i = t0 + lane; i < g.V; i += 32) {
            const float x = VL::scalar(rowp, i);
            if (x >= F) {
                const int pos = atomicAdd(ngather, 1);
                if (pos < GCAP) gbuf[pos] = make_key(x, static_cast<uint32_t>(i));
            }
        }
    }
    __syncwarp();
    {
        const int total = __shfl_sync(FULL, *reinterpret_cast<volatile int *>(ngather), 0);
        if (total <= GCAP) {
            out.clear();
            merge_buffer<R>(out, gbuf, total, lane);
            return out;
        }
    }
    // more elements reach F than the scratch holds: rank every slice
    for (int c = 0; c < g.cpr; ++c) {
        const uint32_t base = static_cast<uint32_t>(c) * CE + lane * VE;
        const bool take = lane * 16 < static_cast<int>(chunk_bulk_bytes(g, c));
        offer_slices<R, BF16>(g, rowp, take, base, true, 0.0f, F, nsel, lane, out, otau);
    }
    // the ragged end
    const int64_t tail0 = static_cast<int64_t>(g.cpr - 1) * CE + chunk_bulk_bytes(g, g.cpr - 1) / esz;
    const int64_t i = tail0 + lane;
    const float x = i < g.V ? VL::scalar(rowp, i) : NEG_INF;
    const bool take = i < g.V && x >= F;
    offer_slices<R, BF16>(g, rowp, take, static_cast<uint32_t>(i < g.V ? i : 0), false, x, F, nsel, lane, out, otau);
    return out;
}

// Warp 0, after scan_row.  A row that lies inside this CTA's range is done:
// returns true.  A row split over several CTAs: publish this CTA's part; the
// CTA that completes the row (per-row ticket) combines the parts in CTA
// order into `res` and returns true, the others return false.
template <int R, int MODE>
__device__ __forceinline__ bool join_parts(const ScanGeom &g, const ScanWs &sw, int64_t row, RowResult<R> &res, float c,
                           int lane) {
    const int64_t b0 = range_owner(g, row * g.cpr);
    const int64_t b1 = range_owner(g, row * g.cpr + g.cpr - 1);
    if (b0 == b1) return true;
    auto rec_of = [&](int64_t bb) -> PartRec * {
        return sw.parts + 2 * bb + (range_begin(g, bb) / g.cpr == row ? 0 : 1);
    };
    PartRec *mine = rec_of(blockIdx.x);
    if (MODE == MODE_ARGMAX) {
        if (lane == 0) mine->keys[0] = res.best;
    } else {
        res.list.store(mine->keys, lane);
    }
    if (lane == 0) {
        mine->m = res.m;
        mine->s = res.s;
        mine->bad = res.bad ? 1 : 0;
    }
    __syncwarp();
    int old = 0;
    if (lane == 0) old = atomic_add_acq_rel(&sw.tickets[row], 1);
    old = __shfl_sync(FULL, old, 0);
    if (old != static_cast<int>(b1 - b0)) return false;
    if (lane == 0) sw.tickets[row] = 0;  // zero again for the next call
    __syncwarp();
    bool bad = false;
    uint64_t best = 0;
    float m = NEG_INF, s = 0.0f;
    WarpList<R> acc;
    acc.clear();
    for (int64_t bb = b0; bb <= b1; ++bb) {
        const PartRec *p = rec_of(bb);
        bad |= __ldcg(&p->bad) != 0;
        if (MODE == MODE_ARGMAX) {
            const uint64_t k = __ldcg(reinterpret_cast<const unsigned long long *>(&p->keys[0]));
            best = k > best ? k : best;
        } else {
            WarpList<R> o;
#pragma unroll
            for (int r = 0; r < R; ++r)
                o.k[r] = __ldcg(reinterpret_cast<const unsigned long long *>(&p->keys[r * 32 + lane]));
            acc.merge(o, lane);
        }
        if (MODE == MODE_TOPN_LSE) lse_combine(m, s, __ldcg(&p->m), __ldcg(&p->s), c);
    }
    res.bad = bad;
    res.best = best;
    res.list = acc;
    res.m = m;
    res.s = s;
    return true;
}

__device__ __forceinline__ void scan_init(ScanSmem &sm) {
    if (threadIdx.x == 0) {
        for (int w = 0; w < SCAN_WARPS; ++w)
            for (int s = 0; s < WSTAGES; ++s) mbar_init(&sm.full[w][s], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.slot_full[s], SCAN_WARPS);
            mbar_init(&sm.slot_empty[s], 1);
        }
        sm.floor_ord[0] = sm.floor_ord[1] = 0;
        sm.nwide = 0;
        for (int w = 0; w < SCAN_WARPS; ++w) {
            sm.ring_head[w] = sm.ring_tail[w] = 0;
            sm.hand[0].ring_end[w] = sm.hand[1].ring_end[w] = 0;
        }
        fence_barrier_init();
    }
    __syncthreads();
}

// CTAs per SM of a scan kernel: three (the streaming warps hold no lists;
// only the completion warp holds the row's list of 32 or 64 keys).  Verify
// with sampling requests keeps two: its completion work per row (filters,
// draws) is the longer part there, and measured faster at two.
template <bool SAMPLED, bool VERIFY = false>
constexpr int scan_min_blocks() { return SAMPLED && VERIFY ? 2 : 3; }

// The CTA's part of row `row`: how many of the warps hold a chunk of it
// (returned) and the first of them (*w0); they follow cyclically.
__device__ __forceinline__ int row_warps(const ScanGeom &g, int64_t row, int64_t begin, int64_t end, int *w0) {
    const int64_t a = row * g.cpr > begin ? row * g.cpr : begin;
    const int64_t b = (row + 1) * g.cpr < end ? (row + 1) * g.cpr : end;
    *w0 = static_cast<int>((a - begin) % SCAN_WARPS);
    return b - a < SCAN_WARPS ? static_cast<int>(b - a) : SCAN_WARPS;
}

// Grid of a scan launch: as many CTAs as fit, at most MAX_SCAN_GRID and at
// most one per chunk.  When the rows alone nearly fill that many CTAs, one CTA
// per row: no row is split, so no row waits for a join at the end.
inline int64_t scan_grid(int per_sm, int sms, int64_t rows, int64_t total) {
    int64_t grid = static_cast<int64_t>(sms) * per_sm;
    if (grid > MAX_SCAN_GRID) grid = MAX_SCAN_GRID;
    if (rows <= grid && rows * 8 >= grid * 7) return rows;
    if (grid > total) grid = total;
    return grid;
}

}  // namespace dfl
