// lmhead.cu -- dflash2_lmhead_topk16: the drafter's LM head and the top-16
// reduction fused, so that the block logits never reach memory.
//
// DFlash 2 proposer issue, "What upstream shipped" item 1 (keep the top-16
// candidates per drafted position) and FreeToken PR 857, "Details"/Runtime
// (16 candidates per slot from the LM head): the candidates and U come from
// logits = h . W^T over the whole vocabulary.  Here that GEMM runs on the
// 5th-generation tensor cores and each 128 x 256 logit tile is reduced in the
// epilogue straight out of tensor memory.
//
// Work split.  The rows are cut into M tiles of 128 and the vocabulary into
// N tiles of 256.  One CTA per SM owns one M tile and a contiguous range of N
// tiles (ranges of the same M tile are the CTAs of one column of the grid).
// For each N tile: TMA stages 128x64 tiles of h and 256x64 tiles of W
// (128-byte swizzle) through a 4-deep mbarrier ring, one thread issues
// tcgen05.mma (kind::f16, bf16 x bf16 -> fp32) into one of two 256-column
// tensor-memory accumulators, and four epilogue warps (one row of the tile per
// thread) drain the other accumulator: running max and sum of exponentials,
// and a sorted list of the row's 16 best logits.  At the end of its range a
// CTA writes, per row, a partial in the layout of dflash2_topk16_shard (the
// range is a vocabulary slice); a second kernel merges the ranges' partials.
//
// Waits are bounded: a timed-out wait sets the error word and the CTA's rows
// come out -1 / NaN.
#include "host.hpp"
#include "common.cuh"
#include "tc.cuh"

namespace dfl {

static __device__ unsigned int g_err_lmhead;

constexpr int LBM = 128;   // rows of a tile (tensor-memory lanes)
constexpr int LBN = 256;   // vocabulary entries of a tile (accumulator columns)
constexpr int LBK = 64;    // hidden elements per stage (one 128-byte swizzle row)
constexpr int LSTAGES = 4;
constexpr int LM_THREADS = 224;  // warps 0-3 epilogue, 4 TMA producer, 5 MMA issuer, 6 L2 prefetch
constexpr int LM_PF = 12;        // k-blocks of W asked of L2 ahead of the producer (~3 us of MMA)
constexpr int LM_TOP = 16;       // candidates kept per row and range
constexpr long long LM_WAIT = 4000000000ll;   // ~2 s
constexpr long long LM_DRAIN = 200000000ll;   // ~0.1 s

struct LmSmem {
    alignas(1024) unsigned char a[LSTAGES][LBM * LBK * 2];
    alignas(1024) unsigned char b[LSTAGES][LBN * LBK * 2];
    uint64_t full[LSTAGES];
    uint64_t empty[LSTAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t done;
    uint32_t tmem_base;
    int abort_flag;
    int issued;  // k-blocks the producer has copied so far
};

static_assert(sizeof(LmSmem) + 1024 <= 227 * 1024, "the LM-head pipeline fits one SM's shared memory");

struct LmArgs {
    int64_t rows, V;
    int kblocks;      // hidden / 64
    int ntiles;       // N tiles of the vocabulary
    int nranges;      // N ranges per M tile (= partials per row)
    int mtiles;       // M tiles
    const char *W;    // the LM head's weight (for the L2 prefetch)
    const dflash2_sampling *params;
    int64_t rows_per_param;
    int32_t *part_idx;  // [nranges, rows, DFLASH2_SHARD_LIST]
    float *part_z;
    float *part_m;      // [nranges, rows]
    float *part_s;
};

__device__ __forceinline__ uint32_t lm_idesc() {
    return (1u << 4)                                   // D: fp32
           | (1u << 7)                                 // A: bf16
           | (1u << 10)                                // B: bf16
           | (static_cast<uint32_t>(LBN >> 3) << 17)   // N / 8
           | (static_cast<uint32_t>(LBM >> 4) << 24);  // M / 16
}

__device__ __forceinline__ void lm_abort(LmSmem &sm) {
    atomicOr(&g_err_lmhead, ERR_WAIT_TIMEOUT);
    *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
}
__device__ __forceinline__ bool lm_aborted(LmSmem &sm) {
    return *reinterpret_cast<volatile int *>(&sm.abort_flag) != 0;
}

// The row's running state: max m and sum s of 2^((z - m) c), and its 16 best
// logits in descending order (ties: the lower id first; ids arrive in
// increasing order, so a later equal value never displaces an earlier one).
struct RowTop {
    float v[LM_TOP];
    int32_t id[LM_TOP];
    float m, s;
    bool nan;
};

__device__ __forceinline__ void row_insert(RowTop &t, float x, int32_t id) {
    t.v[LM_TOP - 1] = x;
    t.id[LM_TOP - 1] = id;
#pragma unroll
    for (int j = LM_TOP - 1; j > 0; --j) {
        if (t.v[j] > t.v[j - 1]) {
            const float tv = t.v[j];
            t.v[j] = t.v[j - 1];
            t.v[j - 1] = tv;
            const int32_t ti = t.id[j];
            t.id[j] = t.id[j - 1];
            t.id[j - 1] = ti;
        }
    }
}

// 32 logits of the row (columns id0 .. id0 + 31 of the vocabulary).
__device__ __forceinline__ void row_take32(RowTop &t, const uint32_t (&bits)[32], int64_t id0, int64_t V, float c) {
    float x[32];
    float cm = NEG_INF;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        x[i] = id0 + i < V ? __uint_as_float(bits[i]) : NEG_INF;
        t.nan |= x[i] != x[i];
        cm = fmaxf(cm, x[i]);
    }
    if (cm > t.m) {
        t.s *= ex2((t.m - cm) * c);
        t.m = cm;
    }
    if (t.m != NEG_INF) {
        const float nm = -t.m * c;
#pragma unroll
        for (int i = 0; i < 32; ++i) t.s += ex2(fmaf(x[i], c, nm));
    }
    if (cm > t.v[LM_TOP - 1]) {  // rare after the first tiles
        uint32_t cand = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (x[i] > t.v[LM_TOP - 1]) cand |= 1u << i;
#pragma unroll 1
        while (cand) {  // in increasing id order, so ties keep the lower id first
            const int i = __ffs(cand) - 1;
            cand &= cand - 1;
            float xi = x[0];
#pragma unroll
            for (int q = 1; q < 32; ++q)
                if (q == i) xi = x[q];
            if (xi > t.v[LM_TOP - 1]) row_insert(t, xi, static_cast<int32_t>(id0 + i));
        }
    }
}

__global__ void __launch_bounds__(LM_THREADS, 1) k_lmhead(const __grid_constant__ CUtensorMap tm_h,
                                                          const __grid_constant__ CUtensorMap tm_w, LmArgs a) {
    extern __shared__ unsigned char raw[];
    LmSmem &sm = *reinterpret_cast<LmSmem *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int mt = blockIdx.x / a.nranges;
    const int rg = blockIdx.x % a.nranges;
    const int t0 = static_cast<int>(static_cast<int64_t>(a.ntiles) * rg / a.nranges);
    const int t1 = static_cast<int>(static_cast<int64_t>(a.ntiles) * (rg + 1) / a.nranges);
    const int nt = t1 - t0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < LSTAGES; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.acc_full[b], 1);
            mbar_init(&sm.acc_empty[b], 4);
        }
        mbar_init(&sm.done, 1);
        sm.abort_flag = 0;
        sm.issued = 0;
        fence_barrier_init();
    }
    if (warp == 5) tmem_alloc(&sm.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    pdl_wait();     // h and W may come from the grids before this one
    pdl_trigger();  // the merge waits for this grid to complete before it reads anything

    if (warp == 4) {
        // TMA producer
        int it = 0;
        if (lane == 0) {
            for (int j = 0; j < nt && !lm_aborted(sm); ++j) {
                for (int kb = 0; kb < a.kblocks; ++kb, ++it) {
                    const int s = it % LSTAGES;
                    if (it >= LSTAGES && !mbar_wait(&sm.empty[s], ((it / LSTAGES) - 1) & 1, LM_WAIT)) {
                        lm_abort(sm);
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.full[s], (LBM + LBN) * LBK * 2);
                    tma_load_2d(sm.a[s], &tm_h, kb * LBK, mt * LBM, &sm.full[s]);
                    tma_load_2d(sm.b[s], &tm_w, kb * LBK, (t0 + j) * LBN, &sm.full[s]);
                    *reinterpret_cast<volatile int *>(&sm.issued) = it + 1;
                }
            }
            // Leave no copy in flight into this CTA's shared memory.
            for (int i = it > LSTAGES ? it - LSTAGES : 0; i < it; ++i)
                mbar_wait(&sm.full[i % LSTAGES], (i / LSTAGES) & 1, LM_DRAIN);
        }
    } else if (warp == 6) {
        // L2 prefetch of W, LM_PF k-blocks ahead of the producer: the copies of
        // a range's W tiles then find them in L2 instead of waiting on HBM.  The
        // range's CTAs (one per M tile) share the work: this CTA takes rows
        // mt, mt + mtiles, ... of each tile's k-block, one 128-byte line each.
        const int total = nt * a.kblocks;
        const int64_t ld = static_cast<int64_t>(a.kblocks) * LBK * 2;  // bytes per W row
        const long long tstart = clock64();
        for (int i = 0; i < total && !lm_aborted(sm); ++i) {
            while (i >= *reinterpret_cast<volatile int *>(&sm.issued) + LM_PF) {
                if (lm_aborted(sm) || clock64() - tstart > LM_WAIT) break;
                __nanosleep(200);
            }
            if (lm_aborted(sm) || clock64() - tstart > LM_WAIT) break;
            const int64_t n0 = static_cast<int64_t>(t0 + i / a.kblocks) * LBN;
            const int kb = i % a.kblocks;
            for (int rr = mt + lane * a.mtiles; rr < LBN; rr += 32 * a.mtiles) {
                const int64_t v = n0 + rr;
                if (v < a.V) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.W + v * ld + kb * LBK * 2));
            }
        }
    } else if (warp == 5) {
        // MMA issuer
        if (lane == 0) {
            const uint32_t idesc = lm_idesc();
            int it = 0;
            for (int j = 0; j < nt && !lm_aborted(sm); ++j) {
                const int b = j & 1;
                if (j >= 2 && !mbar_wait(&sm.acc_empty[b], ((j >> 1) - 1) & 1, LM_WAIT)) {
                    lm_abort(sm);
                    break;
                }
                tc_fence_after();
                bool ok = true;
                for (int kb = 0; kb < a.kblocks; ++kb, ++it) {
                    const int s = it % LSTAGES;
                    if (!mbar_wait(&sm.full[s], (it / LSTAGES) & 1, LM_WAIT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(sm.a[s]);
                    const uint64_t bd = sw128_desc(sm.b[s]);
#pragma unroll
                    for (int k = 0; k < LBK / 16; ++k)  // 16 bf16 = 32 bytes per MMA: +2 in the address field
                        mma_bf16(tmem + static_cast<uint32_t>(b * LBN), ad + 2 * k, bd + 2 * k, idesc, kb > 0 || k > 0);
                    mma_commit(&sm.empty[s]);
                }
                if (!ok) {
                    lm_abort(sm);
                    break;
                }
                mma_commit(&sm.acc_full[b]);
            }
            // Every MMA issued has completed once this commit arrives.
            mma_commit(&sm.done);
            mbar_wait(&sm.done, 0, LM_DRAIN);
        }
    } else {
        // Epilogue: thread = row w*32 + lane of the tile.
        const int r = warp * 32 + lane;
        const int64_t row = static_cast<int64_t>(mt) * LBM + r;
        const RowTask task = decode_row(a.params, (row < a.rows ? row : 0) / a.rows_per_param, a.V, false);
        const float c = LOG2E / task.T;
        RowTop t;
#pragma unroll
        for (int j = 0; j < LM_TOP; ++j) {
            t.v[j] = NEG_INF;
            t.id[j] = -1;
        }
        t.m = NEG_INF;
        t.s = 0.0f;
        t.nan = false;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            const int b = j & 1;
            ok = ok && !lm_aborted(sm) && mbar_wait(&sm.acc_full[b], (j >> 1) & 1, LM_WAIT);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            tc_fence_after();
            const int64_t n0 = static_cast<int64_t>(t0 + j) * LBN;
            const uint32_t base = tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(b * LBN);
#pragma unroll 1
            for (int cc = 0; cc < LBN / 32; ++cc) {
                uint32_t bits[32];
                tmem_ld16_nowait(base + cc * 32, bits);
                tmem_ld16_nowait(base + cc * 32 + 16, bits + 16);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                row_take32(t, bits, n0 + cc * 32, a.V, c);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.acc_empty[b]);
        }
        if (!ok && lane == 0) lm_abort(sm);
        if (row < a.rows) {
            // Rows that need more than 16 candidates (top_k above 16) or the
            // whole row (top_p with top_k off) are not reduced here.
            const bool bad = !ok || t.nan || task.mode == MODE_SKIP || task.nsel > LM_TOP || t.m == INFINITY;
            const bool lse_row = task.mode == MODE_TOPN_LSE;
            const int64_t o = (static_cast<int64_t>(rg) * a.rows + row) * DFLASH2_SHARD_LIST;
#pragma unroll
            for (int i = 0; i < LM_TOP; ++i) {
                const bool has = !bad && t.id[i] >= 0;
                a.part_idx[o + i] = has ? t.id[i] : -1;
                a.part_z[o + i] = has ? t.v[i] : NEG_INF;
            }
#pragma unroll 1
            for (int i = LM_TOP; i < DFLASH2_SHARD_LIST; ++i) {
                a.part_idx[o + i] = -1;
                a.part_z[o + i] = NEG_INF;
            }
            a.part_m[static_cast<int64_t>(rg) * a.rows + row] = bad ? NAN : (lse_row ? t.m : t.v[0]);
            a.part_s[static_cast<int64_t>(rg) * a.rows + row] =
                bad ? NAN : (lse_row && t.m != NEG_INF ? t.s : 0.0f);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, 512);
}

unsigned int read_error_lmhead(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_err_lmhead, sizeof v);
    if (clear) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_err_lmhead, &z, sizeof z);
    }
    return v;
}

// Ranges per M tile: the CTAs fill the SMs once (one CTA per SM).
static int lm_ranges(int64_t rows, int64_t V) {
    const int64_t mtiles = (rows + LBM - 1) / LBM;
    const int64_t ntiles = (V + LBN - 1) / LBN;
    int64_t r = sm_count() / (mtiles > 0 ? mtiles : 1);
    if (r < 1) r = 1;
    if (r > ntiles) r = ntiles;
    if (r > DFLASH2_MAX_SHARDS) r = DFLASH2_MAX_SHARDS;
    return static_cast<int>(r);
}

static size_t lm_ws_bytes(int64_t rows, int nranges) {
    const size_t lists = static_cast<size_t>(nranges) * rows * DFLASH2_SHARD_LIST;
    const size_t per = static_cast<size_t>(nranges) * rows;
    return ((lists * 4 + 255) / 256 + (lists * 4 + 255) / 256 + (per * 4 + 255) / 256 + (per * 4 + 255) / 256) * 256;
}

}  // namespace dfl

using namespace dfl;

extern "C" size_t dflash2_lmhead_topk16_workspace_bytes(int64_t rows, int64_t V) {
    if (rows < 0 || V < NC) return 0;
    return lm_ws_bytes(rows, lm_ranges(rows, V));
}

extern "C" dflash2_status dflash2_lmhead_topk16(const void *h, const void *W, int64_t rows, int64_t hidden, int64_t V,
                                                const dflash2_sampling *params, int64_t rows_per_param,
                                                int32_t *cand_idx, float *cand_U, float *lse, void *ws,
                                                size_t ws_bytes, dflash2_stream stream) {
    if (rows < 0 || hidden < LBK || hidden % LBK != 0 || V < NC || V >= (int64_t(1) << 31) || rows_per_param < 1)
        return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!h || !W || !cand_idx || !cand_U || !lse || !ws || !aligned16(h) || !aligned16(W) || !aligned16(ws) ||
        (params && (reinterpret_cast<uintptr_t>(params) & 3)))
        return DFLASH2_ERR_INVALID_ARG;
    if (rows >= (int64_t(1) << 31) / LBM) return DFLASH2_ERR_UNSUPPORTED;
    const int nranges = lm_ranges(rows, V);
    if (ws_bytes < lm_ws_bytes(rows, nranges)) return DFLASH2_ERR_WORKSPACE;
    LmArgs a;
    a.rows = rows;
    a.V = V;
    a.kblocks = static_cast<int>(hidden / LBK);
    a.ntiles = static_cast<int>((V + LBN - 1) / LBN);
    a.nranges = nranges;
    a.mtiles = static_cast<int>((rows + LBM - 1) / LBM);
    a.W = static_cast<const char *>(W);
    a.params = params;
    a.rows_per_param = rows_per_param;
    const size_t lists = static_cast<size_t>(nranges) * rows * DFLASH2_SHARD_LIST;
    const size_t per = static_cast<size_t>(nranges) * rows;
    char *p = static_cast<char *>(ws);
    a.part_idx = reinterpret_cast<int32_t *>(p);
    p += (lists * 4 + 255) / 256 * 256;
    a.part_z = reinterpret_cast<float *>(p);
    p += (lists * 4 + 255) / 256 * 256;
    a.part_m = reinterpret_cast<float *>(p);
    p += (per * 4 + 255) / 256 * 256;
    a.part_s = reinterpret_cast<float *>(p);
    CUtensorMap tm_h, tm_w;
    if (!make_map_k64(&tm_h, h, static_cast<uint64_t>(hidden), static_cast<uint64_t>(rows), LBM) ||
        !make_map_k64(&tm_w, W, static_cast<uint64_t>(hidden), static_cast<uint64_t>(V), LBN))
        return DFLASH2_ERR_CUDA;
    const int64_t mtiles = (rows + LBM - 1) / LBM;
    const size_t smem = sizeof(LmSmem) + 1024;
    const void *fn = reinterpret_cast<const void *>(&k_lmhead);
    blocks_per_sm(fn, LM_THREADS, smem);  // raises the shared-memory limit once per device
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(mtiles * nranges), 1, 1);
    cfg.blockDim = dim3(LM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_lmhead, tm_h, tm_w, a) != cudaSuccess) return DFLASH2_ERR_CUDA;
    if (after_launch() != DFLASH2_OK) return DFLASH2_ERR_CUDA;
    return launch_merge16(nranges, rows, a.part_idx, a.part_z, a.part_m, a.part_s, V, params, rows_per_param,
                          cand_idx, cand_U, lse, s);
}
