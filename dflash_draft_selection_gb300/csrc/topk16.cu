// topk16.cu -- dflash2_topk16: the 16 best candidates of every drafted
// position and their log-probabilities U under the drafter's distribution.
//
// DFlash 2 proposer issue, "What upstream shipped" item 1 (keep the top-16
// candidates per position; U_t(b) is the unary term of the pair score, read
// here as the drafter's log-softmax); FreeToken PR 857, "Details"/Runtime
// (16 candidates per slot from the LM head).
#include "host.hpp"
#include "rowscan.cuh"
#include "filter.cuh"

namespace dfl {

static __device__ unsigned int g_err_topk;

template <int R>
__device__ void finalize_draft(const RowResult<R> &res, const RowTask &task, int64_t row,
                               int32_t *cand_idx, float *cand_U, float *lse, int lane) {
    const uint64_t k = res.list.k[0];
    const float z = key_val(k);
    int32_t idx = key_idx(k);
    float U = NAN, L = NAN;
    bool bad = res.bad;
    if (task.mode == MODE_TOPN_LSE) {
        if (!bad && isfinite(res.m)) {
            const float lns = logf(res.s);
            L = res.m / task.T + lns;
            U = (z - res.m) / task.T - lns;
        } else {
            bad = true;
        }
    } else {
        const float z0 = __shfl_sync(FULL, z, 0);
        if (!bad && isfinite(z0)) {
            float e[R], ek;
            const int kept = topn_filter<R>(res.list, task, z0, lane, e, &ek);
            const float lnE = logf(ek);
            L = z0 / task.T + lnE;
            U = lane < kept ? (z - z0) / task.T - lnE : NEG_INF;
        } else {
            bad = true;
        }
    }
    if (bad) {
        idx = -1;
        U = NAN;
        L = NAN;
    }
    if (lane < NC) {
        cand_idx[row * NC + lane] = idx;
        cand_U[row * NC + lane] = U;
    }
    if (lane == 0) lse[row] = L;
}

template <int R, bool BF16>
__global__ void __launch_bounds__(SCAN_THREADS, 3) k_topk16(ScanGeom g, int32_t *cand_idx, float *cand_U,
                                                         float *lse) {
    extern __shared__ unsigned char smem_raw[];
    ScanSmem &sm = *reinterpret_cast<ScanSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    constexpr int esz = BF16 ? 2 : 4;
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    scan_init(sm);
    WarpStream ws;
    stream_start<esz>(sm, g, ws, lane);
    int rp = 0;
    for (int64_t row = blockIdx.x; row < g.rows; row += gridDim.x, rp ^= 1) {
        const RowTask task = decode_row(g.params, row / g.rows_per_param, g.V, false);
        RowResult<R> res;
        if (!row_streams(task)) {
            scan_row<R, MODE_ARGMAX, BF16>(sm, g, ws, task, row, rp, true, res, &g_err_topk);
            if (w == 0) {
                if (lane < NC) {
                    cand_idx[row * NC + lane] = -1;
                    cand_U[row * NC + lane] = NAN;
                }
                if (lane == 0) lse[row] = NAN;
            }
            continue;
        }
        if (task.mode == MODE_TOPN_LSE)
            scan_row<R, MODE_TOPN_LSE, BF16>(sm, g, ws, task, row, rp, false, res, &g_err_topk);
        else
            scan_row<R, MODE_TOPN, BF16>(sm, g, ws, task, row, rp, false, res, &g_err_topk);
        if (w == 0) finalize_draft<R>(res, task, row, cand_idx, cand_U, lse, lane);
    }
    if (ws.aborted) stream_drain(sm, ws);
}

template <int R, bool BF16>
static dflash2_status launch_topk16(const ScanGeom &g, int32_t *cand_idx, float *cand_U, float *lse,
                                    cudaStream_t stream) {
    const size_t smem = scan_smem_bytes();
    const void *fn = reinterpret_cast<const void *>(&k_topk16<R, BF16>);
    const int per_sm = blocks_per_sm(fn, SCAN_THREADS, smem);
    int64_t grid = static_cast<int64_t>(sm_count()) * per_sm;
    if (grid > g.rows) grid = g.rows;
    k_topk16<R, BF16><<<static_cast<unsigned>(grid), SCAN_THREADS, smem, stream>>>(g, cand_idx, cand_U, lse);
    return after_launch();
}

unsigned int read_error_topk(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_err_topk, sizeof v);
    if (clear) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_err_topk, &z, sizeof z);
    }
    return v;
}

}  // namespace dfl

using namespace dfl;

extern "C" dflash2_status dflash2_topk16(const void *logits, dflash2_dtype dt, int64_t rows, int64_t V,
                                         int64_t ld, const dflash2_sampling *params,
                                         int64_t rows_per_param, int32_t *cand_idx, float *cand_U,
                                         float *lse, dflash2_stream stream) {
    if (!dtype_ok(dt) || rows < 0 || V < NC || V >= (int64_t(1) << 31) || ld < V || rows_per_param < 1)
        return DFLASH2_ERR_INVALID_ARG;
    const int es = esize(dt);
    if ((ld * es) % 16 != 0) return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!logits || !cand_idx || !cand_U || !lse || !aligned16(logits) || !aligned16(cand_idx) ||
        !aligned16(cand_U) || !aligned16(lse) || (params && (reinterpret_cast<uintptr_t>(params) & 3)))
        return DFLASH2_ERR_INVALID_ARG;
    ScanGeom g;
    g.base = static_cast<const char *>(logits);
    g.ld_bytes = ld * es;
    g.V = V;
    g.rows = rows;
    g.chunks_per_row = static_cast<int>((V * es + CHUNK_BYTES - 1) / CHUNK_BYTES);
    g.params = params;
    g.rows_per_param = rows_per_param;
    g.target = false;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (params == nullptr)
        return dt == DFLASH2_BF16 ? launch_topk16<1, true>(g, cand_idx, cand_U, lse, s)
                                  : launch_topk16<1, false>(g, cand_idx, cand_U, lse, s);
    return dt == DFLASH2_BF16 ? launch_topk16<2, true>(g, cand_idx, cand_U, lse, s)
                              : launch_topk16<2, false>(g, cand_idx, cand_U, lse, s);
}
