// rowscan.cuh -- one-pass streaming reduction of full-vocabulary logit rows.
//
// Both logit streams of the DFlash 2 path (the drafter's block logits for the
// top-16 candidates and U, the target's verify logits for p) are reductions
// of whole vocabulary rows: a running max / sum of exponentials, an argmax,
// or the best N keys.
//
// Work split.  The rows are cut into 4 KB chunks and the flat chunk sequence
// (row-major) is split into one contiguous range per CTA, equal to within a
// chunk, so every CTA streams the same number of bytes whatever the row count.
// A row that straddles two or more ranges is reduced by each of its CTAs; each
// writes a partial result to the workspace and the CTA that completes the row
// (a per-row ticket) combines the parts in CTA order and finishes the row.
//
// Streaming.  Chunk j of a CTA's range belongs to warp j mod 8.  Each warp
// streams its chunks through a private 2-stage shared-memory ring filled by
// 1-D bulk copies (cp.async.bulk) that complete on per-stage mbarriers; the
// warp that consumes a stage refills it, so no cross-warp handshake is needed.
//
// Per chunk, each lane first takes the maximum of its 64 (bf16) elements with
// packed bf16x2 maxima, then (for the log normaliser) its sum of 2^((x-m)c).
// Argmax: only lanes whose maximum beats the warp's best value rescan their
// elements.  Best N keys: elements below a value floor cannot be among the N
// best; the floor is the best of (a) the warp's N-th key, (b) a bound taken
// from the first chunk (the N-th largest lane maximum: at least N elements
// reach it) and (c) the best floor any warp of the CTA has published for the
// row.  Elements at or above the floor are appended to a per-warp candidate
// buffer in shared memory; a full buffer is sorted (bitonic) and merged into
// the warp's register-resident list, which raises the floor.  At the end of a
// row the warp results are merged (bitonic networks) into warp 0.
//
// Waits are bounded: a warp that times out raises the error word, stops
// issuing copies, waits a bounded time for those in flight and flags its rows.
#pragma once

#include "common.cuh"

namespace dfl {

constexpr int CHUNK_BYTES = 4096;
constexpr int WSTAGES = 2;
constexpr int SCAN_WARPS = 8;
constexpr int SCAN_THREADS = SCAN_WARPS * 32;
constexpr int VEC_PER_CHUNK = CHUNK_BYTES / 16;
constexpr int VEC_PER_LANE = VEC_PER_CHUNK / 32;
constexpr int CAND_CAP = 64;          // candidate buffer of a warp (keys)
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
};

// Partial result of a row reduced by several CTAs.
struct PartRec {
    float m, s;     // log normaliser part
    int32_t bad;
    int32_t pad;
    uint64_t keys[DFLASH2_MAX_TOPK];  // best keys, descending (keys[0] = best for an argmax)
};

struct ScanWs {
    int32_t *tickets;  // [rows], zero between calls
    PartRec *parts;    // [2 * MAX_SCAN_GRID]
};

inline size_t scan_ws_tickets_bytes(int64_t rows) {
    return (static_cast<size_t>(rows) * sizeof(int32_t) + 255) / 256 * 256;
}
inline size_t scan_ws_bytes(int64_t rows) {
    return scan_ws_tickets_bytes(rows) + static_cast<size_t>(2 * MAX_SCAN_GRID) * sizeof(PartRec);
}
inline ScanWs scan_ws_at(void *p, int64_t rows) {
    ScanWs w;
    w.tickets = static_cast<int32_t *>(p);
    w.parts = reinterpret_cast<PartRec *>(static_cast<char *>(p) + scan_ws_tickets_bytes(rows));
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
    unsigned int floor_ord[2];  // CTA-wide value floor of the row (ordered bits), by row parity
    int bad[2];
    float wm[SCAN_WARPS];
    float wsum[SCAN_WARPS];
    uint64_t wbest[SCAN_WARPS];
    uint32_t lmax[SCAN_WARPS][32];  // sorted lane maxima of each warp's first chunk of the row (ordered bits)
    uint64_t cand[SCAN_WARPS][CAND_CAP];
    uint64_t lists[SCAN_WARPS][DFLASH2_MAX_TOPK];
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
// Warp w owns the chunks begin + w, begin + w + 8, ... of its CTA's range:
// n_w of them.  The issue side runs WSTAGES chunks ahead of the consume side,
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
            bulk_g2s(sm.buf[w][stage], ws.iss_row + static_cast<int64_t>(ws.iss_c) * CHUNK_BYTES, bytes, bar);
    }
    __syncwarp();
    ++ws.iss_k;
    ws.iss_c += SCAN_WARPS;
    while (ws.iss_c >= g.cpr) {
        ws.iss_c -= g.cpr;
        ws.iss_row += g.ld_bytes;
    }
}

__device__ __forceinline__ void stream_start(ScanSmem &sm, const ScanGeom &g, WarpStream &ws, int64_t begin,
                                             int64_t end, int w, int lane) {
    const int64_t len = end - begin;
    ws.n_w = len > w ? static_cast<int>((len - w + SCAN_WARPS - 1) / SCAN_WARPS) : 0;
    const int64_t f0 = begin + w;
    const int64_t r0 = f0 / g.cpr;
    ws.iss_c = ws.cons_c = static_cast<int>(f0 - r0 * g.cpr);
    ws.iss_row = g.base + r0 * g.ld_bytes;
    ws.cons_r = static_cast<int>(r0 - begin / g.cpr);
    ws.iss_k = ws.cons_k = 0;
    ws.aborted = false;
    for (int i = 0; i < WSTAGES && ws.iss_k < ws.n_w; ++i) stream_issue(sm, g, ws, w, lane);
}

// After a time-out: wait a bounded time for the copies still in flight.
__device__ __forceinline__ void stream_drain(ScanSmem &sm, const WarpStream &ws, int w) {
    for (int k = ws.cons_k; k < ws.iss_k; ++k)
        mbar_wait(&sm.full[w][k % WSTAGES], (k / WSTAGES) & 1, DRAIN_CYCLES);
    __syncwarp();
}

// ------------------------------------------------------------ scan state ----
// A lane slice is what one lane reads of a chunk: vectors lane + 32 q
// (q < 8) of 16 bytes, 64 bf16 or 32 f32 elements.  Its key orders slices by
// their maximum, then by the index of their first element (lower first); the
// ragged end of a row (fewer than 16 bytes) enters as single elements, below
// every slice of the same value.  Bit 31 of the low word tells them apart.
__device__ __forceinline__ uint64_t slice_key(float vmax, uint32_t base) {
    vmax = (vmax == 0.0f) ? 0.0f : vmax;
    return (static_cast<uint64_t>(f2ord(vmax)) << 32) | static_cast<uint32_t>(~base);
}
__device__ __forceinline__ uint64_t tail_key(float x, uint32_t idx) {
    x = (x == 0.0f) ? 0.0f : x;
    return (static_cast<uint64_t>(f2ord(x)) << 32) | (~idx & 0x7fffffffu);
}
__device__ __forceinline__ bool key_is_slice(uint64_t k) { return (static_cast<uint32_t>(k) & 0x80000000u) != 0; }
__device__ __forceinline__ uint32_t key_base(uint64_t k) { return ~static_cast<uint32_t>(k) & 0x7fffffffu; }

template <int R>
struct ScanState {
    float bv;   // argmax: this lane's best value and its id
    int32_t bi;
    float bw;   // argmax: the warp's best value (warp-uniform)
    float m, s0, s1, negmc, c;
    float tau_val;  // value of the warp's N-th slice key (-inf while the list is short); warp-uniform
    float lo;       // value floor: at least N elements of the row reach it; warp-uniform
    int nbuf;       // keys in the warp's candidate buffer
    bool bad;
    WarpList<R> list;  // best slice keys of the warp
};

template <bool BF16>
struct VecLoad;
template <>
struct VecLoad<true> {
    static constexpr int VE = 8;
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
    // NaN-propagating maximum of the 8 values of a 16-byte vector.
    __device__ __forceinline__ static float vmax(const unsigned char *p) {
        const uint4 w = *reinterpret_cast<const uint4 *>(p);
        const uint32_t mm = bmax2_nan(bmax2_nan(w.x, w.y), bmax2_nan(w.z, w.w));
        return fmax_nan(bf16lo(mm), bf16hi(mm));
    }
    // NaN-propagating maximum of this lane's slice (vectors q < nq), packed
    // bf16x2 maxima; -inf when nq == 0.
    __device__ __forceinline__ static float lane_max(const unsigned char *tile, int lane, int nq) {
        uint32_t a = 0xff80ff80u, b = 0xff80ff80u, c = 0xff80ff80u, d = 0xff80ff80u;
        if (nq == VEC_PER_LANE) {
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q) {
                const uint4 w = *reinterpret_cast<const uint4 *>(tile + (lane + q * 32) * 16);
                a = bmax2_nan(a, w.x);
                b = bmax2_nan(b, w.y);
                c = bmax2_nan(c, w.z);
                d = bmax2_nan(d, w.w);
            }
        } else {
            for (int q = 0; q < nq; ++q) {
                const uint4 w = *reinterpret_cast<const uint4 *>(tile + (lane + q * 32) * 16);
                a = bmax2_nan(a, w.x);
                b = bmax2_nan(b, w.y);
                c = bmax2_nan(c, w.z);
                d = bmax2_nan(d, w.w);
            }
        }
        const uint32_t mm = bmax2_nan(bmax2_nan(a, b), bmax2_nan(c, d));
        return fmax_nan(bf16lo(mm), bf16hi(mm));
    }
    // s0 += 2^(x c + negmc) over the even elements, s1 over the odd ones.
    __device__ __forceinline__ static void accumulate(const unsigned char *p, float c, float negmc, float &s0,
                                                      float &s1) {
        const uint4 w = *reinterpret_cast<const uint4 *>(p);
        s0 += ex2(fmaf(bf16lo(w.x), c, negmc));
        s1 += ex2(fmaf(bf16hi(w.x), c, negmc));
        s0 += ex2(fmaf(bf16lo(w.y), c, negmc));
        s1 += ex2(fmaf(bf16hi(w.y), c, negmc));
        s0 += ex2(fmaf(bf16lo(w.z), c, negmc));
        s1 += ex2(fmaf(bf16hi(w.z), c, negmc));
        s0 += ex2(fmaf(bf16lo(w.w), c, negmc));
        s1 += ex2(fmaf(bf16hi(w.w), c, negmc));
    }
    __device__ __forceinline__ static float scalar(const char *row, int64_t i) {
        const unsigned short b = reinterpret_cast<const unsigned short *>(row)[i];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
};
template <>
struct VecLoad<false> {
    static constexpr int VE = 4;
    __device__ __forceinline__ static void unpack(uint4 w, float (&x)[4]) {
        x[0] = __uint_as_float(w.x);
        x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z);
        x[3] = __uint_as_float(w.w);
    }
    __device__ __forceinline__ static float vmax(const unsigned char *p) {
        const float4 f = *reinterpret_cast<const float4 *>(p);
        return fmax_nan(fmax_nan(f.x, f.y), fmax_nan(f.z, f.w));
    }
    __device__ __forceinline__ static float lane_max(const unsigned char *tile, int lane, int nq) {
        float a = NEG_INF, b = NEG_INF;
        if (nq == VEC_PER_LANE) {
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q) {
                const float4 f = *reinterpret_cast<const float4 *>(tile + (lane + q * 32) * 16);
                a = fmax_nan(a, fmax_nan(f.x, f.y));
                b = fmax_nan(b, fmax_nan(f.z, f.w));
            }
        } else {
            for (int q = 0; q < nq; ++q) {
                const float4 f = *reinterpret_cast<const float4 *>(tile + (lane + q * 32) * 16);
                a = fmax_nan(a, fmax_nan(f.x, f.y));
                b = fmax_nan(b, fmax_nan(f.z, f.w));
            }
        }
        return fmax_nan(a, b);
    }
    __device__ __forceinline__ static void accumulate(const unsigned char *p, float c, float negmc, float &s0,
                                                      float &s1) {
        const float4 f = *reinterpret_cast<const float4 *>(p);
        s0 += ex2(fmaf(f.x, c, negmc));
        s1 += ex2(fmaf(f.y, c, negmc));
        s0 += ex2(fmaf(f.z, c, negmc));
        s1 += ex2(fmaf(f.w, c, negmc));
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

// Named barrier 1 over the first `threads` threads that reach it (a multiple
// of 32); barrier 0 is __syncthreads.
__device__ __forceinline__ void named_barrier(int threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

// Publish a value floor for the row to the other warps of the CTA.
__device__ __forceinline__ void publish_floor(ScanSmem &sm, int rp, float v, int lane) {
    if (lane == 0 && v > NEG_INF) atomicMax(&sm.floor_ord[rp], f2ord(v));
}

// Sort the candidate buffer into the list (32 keys at a time) and raise the
// warp's floor to the value of its N-th slice key.
template <int R>
__device__ __forceinline__ void flush_candidates(ScanSmem &sm, ScanState<R> &st, const uint64_t *cand, int nsel,
                                                 int lane, int rp) {
    __syncwarp();
    for (int base = 0; base < st.nbuf; base += 32) {
        const uint64_t k = base + lane < st.nbuf ? cand[base + lane] : 0;
        WarpList<R> o;
        o.k[0] = warp_sort_desc(k, lane);
#pragma unroll
        for (int r = 1; r < R; ++r) o.k[r] = 0;
        st.list.merge(o, lane);
    }
    st.nbuf = 0;
    __syncwarp();
    const uint64_t tw = st.list.at(nsel - 1);
    if (tw != 0 && key_val(tw) > st.tau_val) {
        st.tau_val = key_val(tw);
        publish_floor(sm, rp, st.tau_val, lane);
    }
}

// Append the keys of the lanes with `lf` to the warp's buffer (one per
// lane), flushing it first when they do not fit.  Warp-uniform.
template <int R>
__device__ __forceinline__ void take_slices(ScanSmem &sm, ScanState<R> &st, bool lf, float cmax, uint64_t key,
                                            int nsel, int lane, uint64_t *cand, int rp) {
    uint32_t bal = __ballot_sync(FULL, lf);
    if (st.nbuf + __popc(bal) > CAND_CAP) {
        flush_candidates<R>(sm, st, cand, nsel, lane, rp);
        lf = lf && cmax >= st.tau_val;  // against the raised floor
        bal = __ballot_sync(FULL, lf);
    }
    if (lf) cand[st.nbuf + __popc(bal & ((1u << lane) - 1u))] = key;
    st.nbuf += __popc(bal);
    __syncwarp();
}

// One element of the ragged end of a row (lane 0 holds it); warp-uniform.
template <int R, int MODE>
__device__ __forceinline__ void scan_one(ScanState<R> &st, float x, uint32_t idx, bool valid, int lane) {
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
            st.s0 *= ex2((st.m - x) * st.c);
            st.s1 *= ex2((st.m - x) * st.c);
            st.m = x;
            st.negmc = -x * st.c;
        }
        if (st.m != NEG_INF) st.s0 += ex2(fmaf(x, st.c, st.negmc));
    }
    const bool c = valid && x == x && x >= fmaxf(st.lo, st.tau_val);
    const uint32_t msk = __ballot_sync(FULL, c);
    if (msk) {
        const int l = __ffs(msk) - 1;
        st.list.insert(tail_key(__shfl_sync(FULL, x, l), __shfl_sync(FULL, idx, l)), lane);
    }
}

// First chunk of each warp in the row (modes TOPN*, N <= 32): every warp of
// the row publishes the sorted maxima of its lanes, waits for the others
// (named barrier over the row's `expect` warps, w0 the first of them) and
// merges their lists: at least N elements reach the N-th largest of those
// maxima, a floor from 8 chunks instead of one.  A warp whose chunk did not
// arrive takes part with -inf maxima, so the barrier always completes.
__device__ __forceinline__ void cta_first_floor(ScanSmem &sm, float &lo, float cmax, int nsel, int expect, int w0,
                                                int w, int lane) {
    uint32_t o = f2ord(cmax == cmax ? cmax : NEG_INF);
    o = warp_sort_desc(o, lane);
    sm.lmax[w][lane] = o;
    named_barrier(expect * 32);
#pragma unroll 1
    for (int i = 0; i < expect; ++i) {
        const int u = (w0 + i) % SCAN_WARPS;
        if (u != w) o = warp_merge_desc_u32(o, sm.lmax[u][lane], lane);
    }
    const float f = ord2f(__shfl_sync(FULL, o, nsel - 1));
    lo = fmaxf(lo, f);
}

// One chunk of a row after its lane maxima (`cmax`, `nq` vectors per lane):
// `bulk` bytes at `tile`, first element e0.  Warp-uniform.
template <int R, int MODE, bool BF16>
__device__ __forceinline__ void consume_chunk(ScanSmem &sm, ScanState<R> &st, const unsigned char *tile, int nq,
                                              float cmax, uint32_t e0, int nsel, int w, int lane, int rp) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    if (cmax != cmax) st.bad = true;
    if (MODE == MODE_ARGMAX) {
        const bool f = cmax > st.bw;
        if (f) {  // rare after the first chunks: the lane's new best, in index order
            float t = st.bw;
            for (int q = 0; q < nq; ++q) {
                const int v = lane + q * 32;
                if (VL::vmax(tile + v * 16) > t) {
                    float x[VE];
                    VL::unpack(*reinterpret_cast<const uint4 *>(tile + v * 16), x);
#pragma unroll
                    for (int e = 0; e < VE; ++e) {
                        if (x[e] > t) {
                            t = x[e];
                            st.bv = x[e];
                            st.bi = static_cast<int32_t>(e0 + v * VE + e);
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
            const float sc = ex2((st.m - cmax) * st.c);
            st.s0 *= sc;
            st.s1 *= sc;
            st.m = cmax;
            st.negmc = -cmax * st.c;
        }
        if (st.m != NEG_INF) {
            if (nq == VEC_PER_LANE) {
#pragma unroll 4
                for (int q = 0; q < VEC_PER_LANE; ++q)
                    VL::accumulate(tile + (lane + q * 32) * 16, st.c, st.negmc, st.s0, st.s1);
            } else {
                for (int q = 0; q < nq; ++q)
                    VL::accumulate(tile + (lane + q * 32) * 16, st.c, st.negmc, st.s0, st.s1);
            }
        }
    }
    // The CTA's floor for the row (one read, broadcast).
    uint32_t so = lane == 0 ? *reinterpret_cast<volatile unsigned int *>(&sm.floor_ord[rp]) : 0u;
    so = __shfl_sync(FULL, so, 0);
    if (so != 0) st.lo = fmaxf(st.lo, ord2f(so));
    const bool lf = nq > 0 && cmax >= fmaxf(st.lo, st.tau_val);
    if (__any_sync(FULL, lf))
        take_slices<R>(sm, st, lf, cmax, slice_key(cmax, e0 + lane * VE), nsel, lane, sm.cand[w], rp);
}

__device__ __forceinline__ bool row_streams(const RowTask &t) { return t.mode != MODE_SKIP; }

// Consume the warp's chunks of the CTA's row `rrel` (global row `row`) and
// merge the warps; on return warp 0 holds the CTA's result for the row (best
// slice keys for modes TOPN*).  Every row of the range goes through here
// (rows that need no scan with `skip`), so that the chunk streams stay in
// step.  `rp` is the parity of the row within the CTA's rows; `expect` warps,
// from warp w0 on (cyclically), hold a chunk of it.
template <int R, int MODE, bool BF16>
__device__ __forceinline__ void scan_row(ScanSmem &sm, const ScanGeom &g, WarpStream &ws, const RowTask &task,
                                         int64_t row, int rrel, int rp, int expect, int w0, bool skip,
                                         RowResult<R> &res, unsigned int *err_word) {
    using VL = VecLoad<BF16>;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int CE = CHUNK_BYTES / esz;
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int nsel = task.nsel;

    ScanState<R> st;
    st.bv = NEG_INF;
    st.bi = -1;
    st.bw = NEG_INF;
    st.m = NEG_INF;
    st.s0 = st.s1 = 0.0f;
    st.negmc = 0.0f;
    st.c = LOG2E / task.T;
    st.bad = false;
    st.list.clear();
    st.tau_val = NEG_INF;
    st.lo = NEG_INF;
    st.nbuf = 0;

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
        const unsigned char *tile = sm.buf[w][stage];
        const int bulk = static_cast<int>(chunk_bulk_bytes(g, c));
        int nq = VEC_PER_LANE;
        if (bulk != CHUNK_BYTES) {
            const int nvt = bulk >> 4;  // valid vectors in the chunk
            nq = nvt > lane ? (nvt - lane + 31) >> 5 : 0;
        }
        float cmax = NEG_INF;
        if (ok && !skip) cmax = VL::lane_max(tile, lane, nq);
        if (MODE != MODE_ARGMAX && first && !skip && nsel <= 32 && expect > 1)
            cta_first_floor(sm, st.lo, cmax, nsel, expect, w0, w, lane);
        if (ok && !skip) {
            const uint32_t e0 = static_cast<uint32_t>(c) * CE;
            consume_chunk<R, MODE, BF16>(sm, st, tile, nq, cmax, e0, nsel, w, lane, rp);
            // Ragged end of the row (fewer than 16 bytes), read by lane 0.
            if (c == g.cpr - 1) {
                const char *rbase = g.base + row * g.ld_bytes;
                const int64_t cnt = g.V - e0;
                for (int64_t i = e0 + bulk / esz; i < e0 + cnt; ++i) {
                    const float xi = lane == 0 ? VL::scalar(rbase, i) : NEG_INF;
                    scan_one<R, MODE>(st, xi, static_cast<uint32_t>(i), lane == 0, lane);
                }
            }
        }
        first = false;
        __syncwarp();
        // After a time-out nothing more is issued or waited for (cons_k stays
        // behind iss_k for the drain); the position still advances.
        if (ok) {
            ++ws.cons_k;
            // Refill this stage with the chunk WSTAGES ahead (possibly of a later row).
            if (ws.iss_k < ws.n_w) stream_issue(sm, g, ws, w, lane);
        }
        ws.cons_c += SCAN_WARPS;
        while (ws.cons_c >= g.cpr) {
            ws.cons_c -= g.cpr;
            ++ws.cons_r;
        }
    }
    if (MODE != MODE_ARGMAX && st.nbuf > 0) flush_candidates<R>(sm, st, sm.cand[w], nsel, lane, rp);

    // ---- merge the warps' results into warp 0 ----
    __syncthreads();
    if (threadIdx.x == 0) {
        sm.floor_ord[rp ^ 1] = 0;
        sm.bad[rp ^ 1] = 0;
    }
    if (__any_sync(FULL, st.bad) && lane == 0) sm.bad[rp] = 1;
    if (MODE == MODE_ARGMAX) {
        uint64_t kb = st.bi >= 0 ? make_key(st.bv, static_cast<uint32_t>(st.bi)) : 0;
        kb = warp_max_u64(kb);
        if (lane == 0) sm.wbest[w] = kb;
    } else {
        if (MODE == MODE_TOPN_LSE) {
            float mm = st.m, s = st.s0 + st.s1;
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) {
                const float m2 = __shfl_xor_sync(FULL, mm, d);
                const float s2 = __shfl_xor_sync(FULL, s, d);
                lse_combine(mm, s, m2, s2, st.c);
            }
            if (lane == 0) {
                sm.wm[w] = mm;
                sm.wsum[w] = s;
            }
        }
        st.list.store(sm.lists[w], lane);
    }
    __syncthreads();
    if (MODE != MODE_ARGMAX) {
#pragma unroll
        for (int stride = 1; stride < SCAN_WARPS; stride *= 2) {
            if ((w % (2 * stride)) == 0) {
                WarpList<R> o;
                o.load(sm.lists[w + stride], lane);
                st.list.merge(o, lane);
                if (2 * stride < SCAN_WARPS) st.list.store(sm.lists[w], lane);
            }
            if (2 * stride < SCAN_WARPS) __syncthreads();
        }
    }
    if (w == 0) {
        res.bad = sm.bad[rp] != 0;
        res.list = st.list;
        res.best = 0;
        res.m = NEG_INF;
        res.s = 0.0f;
        if (MODE == MODE_ARGMAX) {
            uint64_t b = 0;
            for (int i = 0; i < SCAN_WARPS; ++i) b = sm.wbest[i] > b ? sm.wbest[i] : b;
            res.best = b;
        }
        if (MODE == MODE_TOPN_LSE) {
            float mm = sm.wm[0], s = sm.wsum[0];
            for (int i = 1; i < SCAN_WARPS; ++i) lse_combine(mm, s, sm.wm[i], sm.wsum[i], st.c);
            res.m = mm;
            res.s = s;
        }
    }
    // The next row's merge overwrites sm.lists and the per-warp slots only
    // after its own first barrier, which warp 0 reaches after reading here.
}

// Offer every element of the slices chosen by this warp's lanes (`take`,
// slice or tail key `k`) that reaches `F` to the element list `out`, one
// element per lane at a time; `otau` is out's N-th key.  Warp-uniform.
template <int R, bool BF16>
__device__ __forceinline__ void offer_slices(const ScanGeom &g, const char *rowp, bool take, uint64_t k, float F,
                                             int nsel, int lane, WarpList<R> &out, uint64_t &otau) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int CE = CHUNK_BYTES / esz;
    uint64_t cm = 0;
    uint32_t base = key_base(k);
    const bool slice = key_is_slice(k);
    if (take) {
        if (slice) {
            const int c = static_cast<int>(base / CE);
            const int lin = static_cast<int>((base % CE) / VE);
            const int bulk = static_cast<int>(chunk_bulk_bytes(g, c));
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q) {
                if ((lin + q * 32) * 16 < bulk) {
                    const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(rowp + static_cast<int64_t>(base + q * 32 * VE) * esz));
                    float x[VE];
                    VL::unpack(v, x);
#pragma unroll
                    for (int e = 0; e < VE; ++e)
                        if (x[e] >= F) cm |= 1ull << (q * VE + e);  // NaN never passes
                }
            }
        } else {
            cm = 1;
        }
    }
    while (__any_sync(FULL, cm != 0)) {
        uint64_t key = 0;
        if (cm) {
            const int b = __ffsll(static_cast<long long>(cm)) - 1;
            cm &= cm - 1;
            if (slice) {
                const uint32_t idx = base + (b / VE) * 32 * VE + (b % VE);
                key = make_key(VL::scalar(rowp, idx), idx);
            } else {
                key = make_key(key_val(k), base);
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

// Warp 0, once per row (modes TOPN*): the N best elements of the row from
// its best slice keys L.  F, the N-th largest slice maximum, is reached by at
// least N elements, so every one of the N best elements lies in a slice whose
// maximum reaches F: re-read those slices and rank their elements.  If the
// list is full with its last key tied at F, slices tied at F may have been
// left out: then rank every slice of the row.  Returns element keys.
template <int R, bool BF16>
__device__ __forceinline__ WarpList<R> extract_topn(const ScanGeom &g, int64_t row, const WarpList<R> &L, int nsel,
                                                 int lane) {
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int CE = CHUNK_BYTES / esz;
    using VL = VecLoad<BF16>;
    const char *rowp = g.base + row * g.ld_bytes;
    const uint64_t kN = L.at(nsel - 1);
    const float F = kN ? key_val(kN) : NEG_INF;
    const uint64_t kL = L.at(R * 32 - 1);
    WarpList<R> out;
    out.clear();
    uint64_t otau = 0;
    if (!(kL != 0 && key_val(kL) == F)) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint64_t k = L.k[r];
            offer_slices<R, BF16>(g, rowp, k != 0 && key_val(k) >= F, k, F, nsel, lane, out, otau);
        }
        return out;
    }
    for (int c = 0; c < g.cpr; ++c) {
        const uint32_t base = static_cast<uint32_t>(c) * CE + lane * VL::VE;
        const bool take = lane * 16 < static_cast<int>(chunk_bulk_bytes(g, c));
        offer_slices<R, BF16>(g, rowp, take, slice_key(F, base), F, nsel, lane, out, otau);
    }
    // the ragged end
    const int64_t tail0 = static_cast<int64_t>(g.cpr - 1) * CE + chunk_bulk_bytes(g, g.cpr - 1) / esz;
    const int64_t i = tail0 + lane;
    const float x = i < g.V ? VL::scalar(rowp, i) : NEG_INF;
    const bool take = i < g.V && x >= F;
    offer_slices<R, BF16>(g, rowp, take, tail_key(x, static_cast<uint32_t>(i < g.V ? i : 0)), F, nsel, lane, out,
                          otau);
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
    __threadfence();
    __syncwarp();
    int old = 0;
    if (lane == 0) old = atomicAdd(&sw.tickets[row], 1);
    old = __shfl_sync(FULL, old, 0);
    if (old != static_cast<int>(b1 - b0)) return false;
    if (lane == 0) sw.tickets[row] = 0;
    __threadfence();
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
        sm.floor_ord[0] = sm.floor_ord[1] = 0;
        sm.bad[0] = sm.bad[1] = 0;
        fence_barrier_init();
    }
    __syncthreads();
}

// CTAs per SM of a scan kernel: three for all-greedy launches, two when
// requests may sample (two-register-row lists and more row modes).
template <bool SAMPLED>
constexpr int scan_min_blocks() { return SAMPLED ? 2 : 3; }

// The CTA's part of row `row`: how many of the warps hold a chunk of it
// (returned) and the first of them (*w0); they follow cyclically.
__device__ __forceinline__ int row_warps(const ScanGeom &g, int64_t row, int64_t begin, int64_t end, int *w0) {
    const int64_t a = row * g.cpr > begin ? row * g.cpr : begin;
    const int64_t b = (row + 1) * g.cpr < end ? (row + 1) * g.cpr : end;
    *w0 = static_cast<int>((a - begin) % SCAN_WARPS);
    return b - a < SCAN_WARPS ? static_cast<int>(b - a) : SCAN_WARPS;
}

// Grid of a scan launch: as many CTAs as fit, at most MAX_SCAN_GRID and at
// most one per chunk.
inline int64_t scan_grid(int per_sm, int sms, int64_t total) {
    int64_t grid = static_cast<int64_t>(sms) * per_sm;
    if (grid > MAX_SCAN_GRID) grid = MAX_SCAN_GRID;
    if (grid > total) grid = total;
    return grid;
}

}  // namespace dfl
