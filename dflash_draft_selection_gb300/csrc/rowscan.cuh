// rowscan.cuh -- one-pass streaming reduction of full-vocabulary logit rows.
//
// Both logit streams of the DFlash 2 path (the drafter's block logits for the
// top-16 candidates and U, the target's verify logits for p) are reductions
// of whole vocabulary rows: a running max / sum of exponentials, an argmax,
// or the best N keys.  A persistent CTA owns whole rows.  One producer warp
// streams 8 KB tiles of the row into a shared-memory ring with 1-D bulk
// copies (cp.async.bulk, completion on mbarriers); eight consumer warps read
// the tiles once and keep, per thread, the running max and sum of
// exponentials (or argmax), and, per warp, a register-resident list of the
// best keys filtered by a CTA-wide threshold.  At the end of a row the warp
// results are merged (bitonic networks) and consumer warp 0 holds the row
// result.  Every wait is bounded: on time-out the CTA raises the error word,
// stops waiting and flags the rows it could not read.
#pragma once

#include "common.cuh"

namespace dfl {

constexpr int TILE_BYTES = 8192;
constexpr int STAGES = 5;
constexpr int CWARPS = 8;
constexpr int CTHREADS = CWARPS * 32;
constexpr int SCAN_THREADS = CTHREADS + 32;
constexpr int VEC_PER_TILE = TILE_BYTES / 16;
constexpr int VEC_PER_THREAD = VEC_PER_TILE / CTHREADS;
constexpr int BAR_CONSUMERS = 1;  // named barrier id of the consumer warps

struct ScanGeom {
    const char *base;  // logits
    int64_t ld_bytes;  // row stride in bytes
    int64_t V;
    int64_t rows;
    int tiles_per_row;
    const dflash2_sampling *params;
    int64_t rows_per_param;
    bool target;
};

struct ScanSmem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    unsigned long long tau[2];
    int abort_flag;
    int bad[2];
    float wm[CWARPS];
    float wsum[CWARPS];
    uint64_t wbest[CWARPS];
    uint64_t lists[CWARPS][64];
    alignas(128) unsigned char tiles[STAGES][TILE_BYTES];
};

template <int R>
struct RowResult {
    WarpList<R> list;  // merged best keys (modes TOPN*)
    uint64_t best;     // best key (MODE_ARGMAX)
    float m, s;        // max and sum of 2^((x - m) c) (MODE_TOPN_LSE)
    bool bad;          // NaN seen or a wait failed
};

// Per-thread scan state for one row.
template <int R>
struct ScanState {
    float bv;
    int32_t bi;
    float m, s0, s1, negmc, c;
    uint64_t tau;
    float tau_val;
    uint32_t tau_idx;
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
    const bool maybe = valid && vmax >= st.tau_val;
    if (!__any_sync(FULL, maybe)) return;
#pragma unroll
    for (int e = 0; e < VE; ++e) {
        const float xe = x[e];
        const uint32_t ie = idx0 + e;
        const bool c = maybe && (xe > st.tau_val || (xe == st.tau_val && ie < st.tau_idx));
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
    const bool c = valid && (x > st.tau_val || (x == st.tau_val && idx < st.tau_idx));
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

// Bytes the bulk copy of tile j moves (the ragged < 16-byte end of a row is
// read by the consumers straight from global memory).
__device__ __forceinline__ uint32_t tile_bulk_bytes(const ScanGeom &g, int j, int esz) {
    const int64_t te = TILE_BYTES / esz;
    int64_t cnt = g.V - static_cast<int64_t>(j) * te;
    if (cnt > te) cnt = te;
    return static_cast<uint32_t>((cnt * esz) & ~static_cast<int64_t>(15));
}

// Producer warp: stream every tile of every row this CTA owns.
template <bool BF16>
__device__ void scan_producer(ScanSmem &sm, const ScanGeom &g, unsigned int *err_word) {
    constexpr int esz = BF16 ? 2 : 4;
    if ((threadIdx.x & 31) != 0) return;
    uint32_t it = 0;
    for (int64_t row = blockIdx.x; row < g.rows; row += gridDim.x) {
        const RowTask task = decode_row(g.params, row / g.rows_per_param, g.V, g.target);
        if (!row_streams(task)) continue;
        const char *rbase = g.base + row * g.ld_bytes;
        for (int j = 0; j < g.tiles_per_row; ++j, ++it) {
            const int stage = it % STAGES;
            if (it >= STAGES) {
                const bool quick = *reinterpret_cast<volatile int *>(&sm.abort_flag) != 0;
                if (!mbar_wait(&sm.empty[stage], ((it / STAGES) & 1) ^ 1, quick ? 0 : 2000000000ull)) {
                    atomicOr(err_word, ERR_WAIT_TIMEOUT);
                    *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
                }
            }
            const uint32_t bytes = tile_bulk_bytes(g, j, esz);
            mbar_arrive_expect_tx(&sm.full[stage], bytes);
            if (bytes) bulk_g2s(sm.tiles[stage], rbase + static_cast<int64_t>(j) * TILE_BYTES, bytes,
                                &sm.full[stage]);
        }
    }
    // Drain: do not leave copies in flight into this CTA's shared memory.
    const uint32_t first = it > STAGES ? it - STAGES : 0;
    for (uint32_t t = first; t < it; ++t) mbar_wait(&sm.full[t % STAGES], (t / STAGES) & 1, 100000000ull);
}

// Consumer warps: scan one row; on return consumer warp 0 holds the result.
// `it` is the CTA's running tile counter, `rp` the parity of this row among
// the rows the CTA scanned.
template <int R, int MODE, bool BF16>
__device__ void scan_row(ScanSmem &sm, const ScanGeom &g, const RowTask &task, int64_t row,
                         uint32_t &it, int rp, RowResult<R> &res, unsigned int *err_word) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int TE = TILE_BYTES / esz;
    const int lane = threadIdx.x & 31;
    const int cw = (threadIdx.x >> 5) - 1;
    const int ctid = cw * 32 + lane;
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

    const char *rbase = g.base + row * g.ld_bytes;
    for (int j = 0; j < g.tiles_per_row; ++j, ++it) {
        const int stage = it % STAGES;
        const bool quick = *reinterpret_cast<volatile int *>(&sm.abort_flag) != 0;
        const bool ok = mbar_wait(&sm.full[stage], (it / STAGES) & 1, quick ? 0 : 2000000000ull);
        if (!ok) {
            st.bad = true;
            if (lane == 0) {
                atomicOr(err_word, ERR_WAIT_TIMEOUT);
                *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
            }
        }
        if (MODE != MODE_ARGMAX) {
            const uint64_t shared_tau = *reinterpret_cast<volatile unsigned long long *>(&sm.tau[rp]);
            if (shared_tau > st.tau) st.set_tau(shared_tau);
        }
        const int64_t e0 = static_cast<int64_t>(j) * TE;
        int64_t cnt = g.V - e0;
        if (cnt > TE) cnt = TE;
        const int bulk = static_cast<int>((cnt * esz) & ~static_cast<int64_t>(15));
        const unsigned char *tile = sm.tiles[stage];
#pragma unroll
        for (int q = 0; q < VEC_PER_THREAD; ++q) {
            const int v = ctid + q * CTHREADS;
            const bool valid = ok && v * 16 < bulk;
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
        // Ragged end of the row (fewer than 16 bytes): consumer warp 0, lane 0.
        if (cw == 0 && bulk < cnt * esz) {
            for (int64_t i = e0 + bulk / esz; i < e0 + cnt; ++i) {
                const float xi = lane == 0 ? VL::scalar(rbase, i) : NEG_INF;
                scan_one<R, MODE>(st, xi, static_cast<uint32_t>(i), lane == 0 && ok, nsel, lane);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
        if (MODE != MODE_ARGMAX && lane == 0 && st.tau != 0)
            atomicMax(&sm.tau[rp], static_cast<unsigned long long>(st.tau));
    }

    // ---- merge the warps' results into consumer warp 0 ----
    named_bar_sync(BAR_CONSUMERS, CTHREADS);  // A
    if (ctid == 0) {
        sm.tau[rp ^ 1] = 0;
        sm.bad[rp ^ 1] = 0;
    }
    if (__any_sync(FULL, st.bad) && lane == 0) sm.bad[rp] = 1;
    if (MODE == MODE_ARGMAX) {
        uint64_t k = st.bi >= 0 ? make_key(st.bv, static_cast<uint32_t>(st.bi)) : 0;
        k = warp_max_u64(k);
        if (lane == 0) sm.wbest[cw] = k;
    } else {
        if (MODE == MODE_TOPN_LSE) {
            float m = st.m, s = st.s0 + st.s1;
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) {
                const float m2 = __shfl_xor_sync(FULL, m, d);
                const float s2 = __shfl_xor_sync(FULL, s, d);
                lse_combine(m, s, m2, s2, st.c);
            }
            if (lane == 0) {
                sm.wm[cw] = m;
                sm.wsum[cw] = s;
            }
        }
        st.list.store(sm.lists[cw], lane);
    }
    named_bar_sync(BAR_CONSUMERS, CTHREADS);  // B
    if (MODE != MODE_ARGMAX) {
        WarpList<R> o;
        if ((cw & 1) == 0) {
            o.load(sm.lists[cw + 1], lane);
            st.list.merge(o, lane);
            st.list.store(sm.lists[cw], lane);
        }
        named_bar_sync(BAR_CONSUMERS, CTHREADS);
        if ((cw & 3) == 0) {
            o.load(sm.lists[cw + 2], lane);
            st.list.merge(o, lane);
            st.list.store(sm.lists[cw], lane);
        }
        named_bar_sync(BAR_CONSUMERS, CTHREADS);
        if (cw == 0) {
            o.load(sm.lists[4], lane);
            st.list.merge(o, lane);
        }
    }
    if (cw == 0) {
        res.bad = sm.bad[rp] != 0;
        res.list = st.list;
        res.best = 0;
        res.m = NEG_INF;
        res.s = 0.0f;
        if (MODE == MODE_ARGMAX) {
            uint64_t b = 0;
            for (int w = 0; w < CWARPS; ++w) b = sm.wbest[w] > b ? sm.wbest[w] : b;
            res.best = b;
        }
        if (MODE == MODE_TOPN_LSE) {
            float m = sm.wm[0], s = sm.wsum[0];
            for (int w = 1; w < CWARPS; ++w) lse_combine(m, s, sm.wm[w], sm.wsum[w], st.c);
            res.m = m;
            res.s = s;
        }
    }
}

__device__ __forceinline__ void scan_init(ScanSmem &sm) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], CWARPS);
        }
        sm.tau[0] = sm.tau[1] = 0;
        sm.bad[0] = sm.bad[1] = 0;
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
}

}  // namespace dfl
