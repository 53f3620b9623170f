// rowscan.cuh -- one-pass streaming reduction of full-vocabulary logit rows.
//
// Both logit streams of the DFlash 2 path (the drafter's block logits for the
// top-16 candidates and U, the target's verify logits for p) are reductions
// of whole vocabulary rows: a running max / sum of exponentials, an argmax,
// or the best N keys.  A persistent CTA of 8 warps owns whole rows.  Each
// warp streams its own interleaved 2 KB chunks of the row (chunk c belongs to
// warp c mod 8) through a private 4-stage shared-memory ring filled by 1-D
// bulk copies (cp.async.bulk) that complete on per-stage mbarriers; the warp
// that consumes a stage is the one that refills it, so no cross-warp
// handshake is needed.  Each thread keeps the running max and sum of
// exponentials (or argmax) of its elements, each warp a register-resident
// list of its best keys filtered by a CTA-wide threshold value.  At the end of a
// row the warp results are merged (bitonic networks) and warp 0 holds the
// row result.  Waits are bounded: a warp that times out raises the error
// word, stops issuing copies, waits a bounded time for those in flight and
// flags its rows.
#pragma once

#include "common.cuh"

namespace dfl {

constexpr int CHUNK_BYTES = 2048;
constexpr int WSTAGES = 4;
constexpr int SCAN_WARPS = 8;
constexpr int SCAN_THREADS = SCAN_WARPS * 32;
constexpr int VEC_PER_CHUNK = CHUNK_BYTES / 16;
constexpr int VEC_PER_LANE = VEC_PER_CHUNK / 32;
constexpr long long WAIT_CYCLES = 4000000000ll;  // ~2 s at 2 GHz
constexpr long long DRAIN_CYCLES = 200000000ll;  // ~0.1 s

struct ScanGeom {
    const char *base;  // logits
    int64_t ld_bytes;  // row stride in bytes
    int64_t V;
    int64_t rows;
    int chunks_per_row;
    const dflash2_sampling *params;
    int64_t rows_per_param;
    bool target;
};

struct ScanSmem {
    uint64_t full[SCAN_WARPS][WSTAGES];
    unsigned int tau_ord[2];  // CTA-wide threshold: ordered value bits of the best warp's N-th key
    int bad[2];
    float wm[SCAN_WARPS];
    float wsum[SCAN_WARPS];
    uint64_t wbest[SCAN_WARPS];
    uint64_t lists[SCAN_WARPS][64];
    alignas(128) unsigned char buf[SCAN_WARPS][WSTAGES][CHUNK_BYTES];
};

constexpr size_t scan_smem_bytes() { return sizeof(ScanSmem) + 128; }

template <int R>
struct RowResult {
    WarpList<R> list;  // merged best keys (modes TOPN*)
    uint64_t best;     // best key (MODE_ARGMAX)
    float m, s;        // max and sum of 2^((x - m) c) (MODE_TOPN_LSE)
    bool bad;          // NaN seen or a wait failed
};

// ------------------------------------------------------ per-warp streams ----
// Item k of warp w is chunk w + 8 (k mod n_w) of the CTA's (k / n_w)-th row.
struct WarpStream {
    int w;          // warp index
    int n_w;        // chunks per row owned by this warp
    int64_t total;  // items over all rows of this CTA
    int64_t issued;
    int64_t consumed;
    bool aborted;
};

__device__ __forceinline__ uint32_t chunk_bulk_bytes(const ScanGeom &g, int c, int esz) {
    int64_t bytes = g.V * esz - static_cast<int64_t>(c) * CHUNK_BYTES;
    if (bytes > CHUNK_BYTES) bytes = CHUNK_BYTES;
    return static_cast<uint32_t>(bytes & ~static_cast<int64_t>(15));
}

// Lane 0 issues item k of the warp's stream into its stage.
template <int ESZ>
__device__ __forceinline__ void stream_issue(ScanSmem &sm, const ScanGeom &g, WarpStream &ws, int64_t k,
                                             int lane) {
    const int stage = static_cast<int>(k % WSTAGES);
    const int64_t row = blockIdx.x + (k / ws.n_w) * gridDim.x;
    const int c = ws.w + SCAN_WARPS * static_cast<int>(k % ws.n_w);
    if (lane == 0) {
        const uint32_t bytes = chunk_bulk_bytes(g, c, ESZ);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&sm.full[ws.w][stage], bytes);
        if (bytes)
            bulk_g2s(sm.buf[ws.w][stage], g.base + row * g.ld_bytes + static_cast<int64_t>(c) * CHUNK_BYTES,
                     bytes, &sm.full[ws.w][stage]);
    }
    __syncwarp();
}

template <int ESZ>
__device__ __forceinline__ void stream_start(ScanSmem &sm, const ScanGeom &g, WarpStream &ws, int lane) {
    ws.w = threadIdx.x >> 5;
    ws.n_w = ws.w < g.chunks_per_row ? (g.chunks_per_row - ws.w + SCAN_WARPS - 1) / SCAN_WARPS : 0;
    const int64_t my_rows = blockIdx.x < g.rows ? (g.rows - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    ws.total = my_rows * ws.n_w;
    ws.issued = 0;
    ws.consumed = 0;
    ws.aborted = false;
    while (ws.issued < ws.total && ws.issued < WSTAGES) stream_issue<ESZ>(sm, g, ws, ws.issued++, lane);
}

// After a time-out: wait a bounded time for the copies still in flight.
__device__ __forceinline__ void stream_drain(ScanSmem &sm, WarpStream &ws) {
    for (int64_t k = ws.consumed; k < ws.issued; ++k)
        mbar_wait(&sm.full[ws.w][k % WSTAGES], static_cast<uint32_t>((k / WSTAGES) & 1), DRAIN_CYCLES);
    __syncwarp();
}

// ------------------------------------------------------------ scan state ----
template <int R>
struct ScanState {
    float bv;
    int32_t bi;
    float m, s0, s1, negmc, c;
    uint64_t tau;     // this warp's N-th best key (0 while the list is short)
    float tau_val;
    uint32_t tau_idx;
    float sval;       // CTA-wide threshold value: no element below it can be in the top N
    bool bad;
    WarpList<R> list;

    __device__ __forceinline__ void set_tau(uint64_t t) {
        tau = t;
        if (t == 0) {
            tau_val = NEG_INF;
            tau_idx = 0xffffffffu;
        } else {
            tau_val = key_val(t);
            tau_idx = static_cast<uint32_t>(key_idx(t));
        }
    }
};

// Offer the elements x[0..VE) (token ids idx0 + e) of one vector to the warp
// list.  `valid` may differ across lanes; the call is warp-uniform.
template <int R, int VE>
__device__ __forceinline__ void offer_topn(ScanState<R> &st, const float (&x)[VE], float vmax,
                                           uint32_t idx0, bool valid, int nsel, int lane) {
    const bool maybe = valid && vmax >= fmaxf(st.tau_val, st.sval);
    if (!__any_sync(FULL, maybe)) return;
#pragma unroll
    for (int e = 0; e < VE; ++e) {
        const float xe = x[e];
        const uint32_t ie = idx0 + e;
        const bool c = maybe && xe >= st.sval && (xe > st.tau_val || (xe == st.tau_val && ie < st.tau_idx));
        uint32_t msk = __ballot_sync(FULL, c);
        while (msk) {
            const int l = __ffs(msk) - 1;
            msk &= msk - 1;
            const float xv = __shfl_sync(FULL, xe, l);
            const uint32_t iv = __shfl_sync(FULL, ie, l);
            const uint64_t key = make_key(xv, iv);
            if (key > st.tau) {
                st.list.insert(key, lane);
                const uint64_t tw = st.list.at(nsel - 1);
                if (tw > st.tau) st.set_tau(tw);
            }
        }
    }
}

template <int R, int MODE, int VE>
__device__ __forceinline__ void scan_vec(ScanState<R> &st, const float (&x)[VE], float vmax,
                                         uint32_t idx0, bool valid, int nsel, int lane) {
    if (valid && vmax != vmax) st.bad = true;
    if (MODE == MODE_ARGMAX) {
        if (valid && vmax > st.bv) {
#pragma unroll
            for (int e = 0; e < VE; ++e)
                if (x[e] > st.bv) {
                    st.bv = x[e];
                    st.bi = static_cast<int32_t>(idx0 + e);
                }
        }
    } else {
        if (MODE == MODE_TOPN_LSE && valid) {
            if (vmax > st.m) {
                st.s0 *= ex2((st.m - vmax) * st.c);
                st.s1 *= ex2((st.m - vmax) * st.c);
                st.m = vmax;
                st.negmc = -vmax * st.c;
            }
            if (st.m != NEG_INF) {
#pragma unroll
                for (int e = 0; e < VE; e += 2) {
                    st.s0 += ex2(fmaf(x[e], st.c, st.negmc));
                    st.s1 += ex2(fmaf(x[e + 1], st.c, st.negmc));
                }
            }
        }
        offer_topn<R, VE>(st, x, vmax, idx0, valid, nsel, lane);
    }
}

// One element (only lanes with `valid` hold one); warp-uniform.
template <int R, int MODE>
__device__ __forceinline__ void scan_one(ScanState<R> &st, float x, uint32_t idx, bool valid,
                                         int nsel, int lane) {
    if (valid && x != x) st.bad = true;
    if (MODE == MODE_ARGMAX) {
        if (valid && x > st.bv) {
            st.bv = x;
            st.bi = static_cast<int32_t>(idx);
        }
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
    const bool c = valid && x >= st.sval && (x > st.tau_val || (x == st.tau_val && idx < st.tau_idx));
    uint32_t msk = __ballot_sync(FULL, c);
    while (msk) {
        const int l = __ffs(msk) - 1;
        msk &= msk - 1;
        const uint64_t key = make_key(__shfl_sync(FULL, x, l), __shfl_sync(FULL, idx, l));
        if (key > st.tau) {
            st.list.insert(key, lane);
            const uint64_t tw = st.list.at(nsel - 1);
            if (tw > st.tau) st.set_tau(tw);
        }
    }
}

template <bool BF16>
struct VecLoad;
template <>
struct VecLoad<true> {
    static constexpr int VE = 8;
    __device__ __forceinline__ static void load(const unsigned char *p, float (&x)[8], float &vmax) {
        const uint4 w = *reinterpret_cast<const uint4 *>(p);
        const uint32_t mm = bmax2_nan(bmax2_nan(w.x, w.y), bmax2_nan(w.z, w.w));
        vmax = fmax_nan(bf16lo(mm), bf16hi(mm));
        x[0] = bf16lo(w.x);
        x[1] = bf16hi(w.x);
        x[2] = bf16lo(w.y);
        x[3] = bf16hi(w.y);
        x[4] = bf16lo(w.z);
        x[5] = bf16hi(w.z);
        x[6] = bf16lo(w.w);
        x[7] = bf16hi(w.w);
    }
    __device__ __forceinline__ static float scalar(const char *row, int64_t i) {
        const unsigned short b = reinterpret_cast<const unsigned short *>(row)[i];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
};
template <>
struct VecLoad<false> {
    static constexpr int VE = 4;
    __device__ __forceinline__ static void load(const unsigned char *p, float (&x)[4], float &vmax) {
        const float4 f = *reinterpret_cast<const float4 *>(p);
        x[0] = f.x;
        x[1] = f.y;
        x[2] = f.z;
        x[3] = f.w;
        vmax = fmax_nan(fmax_nan(f.x, f.y), fmax_nan(f.z, f.w));
    }
    __device__ __forceinline__ static float scalar(const char *row, int64_t i) {
        return reinterpret_cast<const float *>(row)[i];
    }
};

__device__ __forceinline__ bool row_streams(const RowTask &t) { return t.mode != MODE_SKIP; }

// Consume the warp's chunks of one row of the CTA (global row `row`) and
// merge the warps; on return warp 0 holds the result.  Every row of the CTA
// goes through here (rows that need no scan with `skip`), so that the chunk
// streams stay in step.  `rp` is the parity of this row among the CTA's rows.
template <int R, int MODE, bool BF16>
__device__ void scan_row(ScanSmem &sm, const ScanGeom &g, WarpStream &ws, const RowTask &task, int64_t row,
                         int rp, bool skip, RowResult<R> &res, unsigned int *err_word) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int CE = CHUNK_BYTES / esz;
    const int lane = threadIdx.x & 31;
    const int w = ws.w;
    const int nsel = task.nsel;

    ScanState<R> st;
    st.bv = NEG_INF;
    st.bi = -1;
    st.m = NEG_INF;
    st.s0 = st.s1 = 0.0f;
    st.negmc = 0.0f;
    st.c = LOG2E / task.T;
    st.bad = false;
    st.list.clear();
    st.set_tau(0);
    st.sval = NEG_INF;

    const char *rbase = g.base + row * g.ld_bytes;
    for (int m = 0; m < ws.n_w; ++m) {
        const int64_t k = ws.consumed;
        const int stage = static_cast<int>(k % WSTAGES);
        bool ok = !ws.aborted && mbar_wait(&sm.full[w][stage], static_cast<uint32_t>((k / WSTAGES) & 1),
                                           WAIT_CYCLES);
        ok = __all_sync(FULL, ok);
        if (!ok && !ws.aborted) {
            ws.aborted = true;
            if (lane == 0) atomicOr(err_word, ERR_WAIT_TIMEOUT);
        }
        if (!ok) st.bad = true;
        if (ok) ws.consumed = k + 1;
        const int c = w + SCAN_WARPS * m;
        if (ok && !skip) {
            if (MODE != MODE_ARGMAX) {
                const uint32_t so = *reinterpret_cast<volatile unsigned int *>(&sm.tau_ord[rp]);
                if (so != 0) st.sval = fmaxf(st.sval, ord2f(so));
            }
            const int64_t e0 = static_cast<int64_t>(c) * CE;
            int64_t cnt = g.V - e0;
            if (cnt > CE) cnt = CE;
            const int bulk = static_cast<int>((cnt * esz) & ~static_cast<int64_t>(15));
            const unsigned char *tile = sm.buf[w][stage];
#pragma unroll
            for (int q = 0; q < VEC_PER_LANE; ++q) {
                const int v = lane + q * 32;
                const bool valid = v * 16 < bulk;
                float x[VE];
                float vmax = NEG_INF;
                if (valid) {
                    VL::load(tile + v * 16, x, vmax);
                } else {
#pragma unroll
                    for (int e = 0; e < VE; ++e) x[e] = NEG_INF;
                }
                scan_vec<R, MODE, VE>(st, x, vmax, static_cast<uint32_t>(e0 + v * VE), valid, nsel, lane);
            }
            // Ragged end of the row (fewer than 16 bytes), read by lane 0.
            if (bulk < cnt * esz) {
                for (int64_t i = e0 + bulk / esz; i < e0 + cnt; ++i) {
                    const float xi = lane == 0 ? VL::scalar(rbase, i) : NEG_INF;
                    scan_one<R, MODE>(st, xi, static_cast<uint32_t>(i), lane == 0, nsel, lane);
                }
            }
            // Publish the warp's N-th value (32-bit: a native shared-memory max).
            if (MODE != MODE_ARGMAX && lane == 0 && st.tau != 0)
                atomicMax(&sm.tau_ord[rp], static_cast<uint32_t>(st.tau >> 32));
        }
        __syncwarp();
        // Refill this stage with the item WSTAGES ahead (possibly of the next row).
        if (ok && ws.issued < ws.total) stream_issue<esz>(sm, g, ws, ws.issued++, lane);
    }

    // ---- merge the warps' results into warp 0 ----
    __syncthreads();  // A
    if (threadIdx.x == 0) {
        sm.tau_ord[rp ^ 1] = 0;
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
    __syncthreads();  // B
    if (MODE != MODE_ARGMAX) {
        WarpList<R> o;
        if ((w & 1) == 0) {
            o.load(sm.lists[w + 1], lane);
            st.list.merge(o, lane);
            st.list.store(sm.lists[w], lane);
        }
        __syncthreads();
        if ((w & 3) == 0) {
            o.load(sm.lists[w + 2], lane);
            st.list.merge(o, lane);
            st.list.store(sm.lists[w], lane);
        }
        __syncthreads();
        if (w == 0) {
            o.load(sm.lists[4], lane);
            st.list.merge(o, lane);
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
}

__device__ __forceinline__ void scan_init(ScanSmem &sm) {
    if (threadIdx.x == 0) {
        for (int w = 0; w < SCAN_WARPS; ++w)
            for (int s = 0; s < WSTAGES; ++s) mbar_init(&sm.full[w][s], 1);
        sm.tau_ord[0] = sm.tau_ord[1] = 0;
        sm.bad[0] = sm.bad[1] = 0;
        fence_barrier_init();
    }
    __syncthreads();
}

}  // namespace dfl
