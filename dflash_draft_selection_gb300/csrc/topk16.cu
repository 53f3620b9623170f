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
#include "wide.cuh"

namespace dfl {

static __device__ unsigned int g_err_topk;

// The row's candidates, U and lse.  A wide row (wc non-NULL) keeps the first
// wc->cut tokens in the order key, of mass wc->P relative to the row maximum.
template <int R>
__device__ __forceinline__ void finalize_draft(const RowResult<R> &res, const RowTask &task, int64_t row,
                               int32_t *cand_idx, float *cand_U, float *lse, int lane,
                               const WideCut *wc = nullptr) {
    const uint64_t k = res.list.k[0];
    const float z = key_val(k);
    int32_t idx = key_idx(k);
    float U = NAN, L = NAN;
    bool bad = res.bad;
    if (task.mode == MODE_TOPN_LSE) {
        if (!bad && isfinite(res.m)) {
            const float lns = logf(wc ? wc->P : res.s);
            L = res.m / task.T + lns;
            U = (z - res.m) / task.T - lns;
            if (wc && lane >= wc->cut) U = NEG_INF;
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

// A wide row whose cut needs passes over the row is left to the CTA's
// epilogue: its ids go out now, its logits (in cand_U) and maximum (in lse)
// until then, and the row is marked as this CTA's.
template <int R>
__device__ __forceinline__ void defer_draft(ScanSmem &sm, const ScanWs &sw, const RowResult<R> &res, int64_t row,
                                            int32_t *cand_idx, float *cand_U, float *lse, int lane) {
    const uint64_t k = res.list.k[0];
    if (lane < NC) {
        cand_idx[row * NC + lane] = key_idx(k);
        cand_U[row * NC + lane] = key_val(k);
    }
    if (lane == 0) {
        lse[row] = res.m;
        sw.marks[row] = static_cast<int32_t>(blockIdx.x) + 1;
        ++sm.nwide;
    }
}

// The epilogue's outputs of a marked row (as finalize_draft writes them).
__device__ __forceinline__ void finalize_deferred(const RowTask &task, int64_t row, float m, const WideCut &wc,
                                                  float *cand_U, float *lse, int lane) {
    const float lns = logf(wc.P);
    if (lane < NC) {
        const float z = cand_U[row * NC + lane];
        cand_U[row * NC + lane] = lane < wc.cut ? (z - m) / task.T - lns : NEG_INF;
    }
    if (lane == 0) lse[row] = m / task.T + lns;
}

// A completed row whose filter may reach past its 64 best: the cut from the
// list when it decides it, else the row is left to the epilogue.
template <int R, bool BF16>
__device__ __forceinline__ void draft_wide_done(ScanSmem &sm, const ScanGeom &g, const ScanWs &sw,
                                                const RowResult<R> &res, const RowTask &task, int64_t row,
                                                int32_t *cand_idx, float *cand_U, float *lse, int lane) {
    WideCut wc;
    wc.cut = 0;
    wc.P = NAN;
    if constexpr (R == 2) {
        if (!res.bad && isfinite(res.m) &&
            !wide_cut_list<BF16>(res.list, res.m, res.s, LOG2E / task.T, task.ek, task.top_p, g.V, &wc, lane)) {
            defer_draft<R>(sm, sw, res, row, cand_idx, cand_U, lse, lane);
            return;
        }
    }
    finalize_draft<R>(res, task, row, cand_idx, cand_U, lse, lane, &wc);
}

// The rows this CTA marked, on all five warps once the CTA has streamed its
// range: the cut by passes over the row, then the row's U and lse.
template <bool BF16>
__device__ __forceinline__ void draft_epilogue(ScanSmem &ssm, const ScanGeom g, const ScanWs sw, int64_t r_first,
                                            int64_t r_last, float *cand_U, float *lse) {
    WideSmem &sm = wide_smem(ssm);
    const Team tm{static_cast<int>(threadIdx.x), SCAN_THREADS};
    const int lane = threadIdx.x & 31;
    const int32_t me = static_cast<int32_t>(blockIdx.x) + 1;
    for (int64_t row = r_first; row <= r_last; ++row) {
        if (sw.marks[row] != me) continue;  // the same for every thread: only this CTA writes `me`
        const RowTask task = decode_row(g.params, row / g.rows_per_param, g.V_params, false);
        const float m = lse[row];
        const WideCut wc = wide_cut_passes<BF16>(tm, sm, g, row, m, LOG2E / task.T, task.ek, task.top_p, lane);
        if (tm.warp() == 0) finalize_deferred(task, row, m, wc, cand_U, lse, lane);
        tm.sync();
        if (threadIdx.x == 0) sw.marks[row] = 0;
    }
}

// Outputs of a vocabulary shard's partial (dflash2_topk16_shard); part_idx
// NULL for the ordinary call.
struct ShardOut {
    int32_t *part_idx;  // [rows, DFLASH2_SHARD_LIST] global ids, -1 past the row's list
    float *part_z;      // [rows, DFLASH2_SHARD_LIST] logits, -inf past the list
    float *part_m;      // [rows] the shard's largest logit
    float *part_s;      // [rows] sum of exp((z - m) / T') over the shard (0 for filtered rows)
    int64_t id_offset;  // global id of the shard's token 0
};

// A shard row's partial: its list's first nsel keys as (global id, logit),
// the largest logit and the sum of the log normaliser; a row with a NaN or
// +Inf, bad or unsupported parameters gets -1 ids, m and s NaN.  A slice of
// masked tokens (every logit -inf) keeps its list, with m = -inf and s = 0.
// Warp-uniform.
template <int R>
__device__ __forceinline__ void finalize_shard(const RowResult<R> &res, const RowTask &task, int64_t row,
                                               const ShardOut &so, int lane) {
    const float top = __shfl_sync(FULL, key_val(res.list.k[0]), 0);
    const float m = task.mode == MODE_TOPN_LSE ? res.m : top;
    // a wide row's filter needs the whole row: not a partial's job
    const bool bad = res.bad || task.mode == MODE_SKIP || task.mode == MODE_ARGMAX || task.wide || m != m ||
                     m == INFINITY;
#pragma unroll
    for (int r = 0; r < DFLASH2_SHARD_LIST / 32; ++r) {
        const int p = r * 32 + lane;
        uint64_t k = 0;
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
            if (rr == r) k = res.list.k[rr];
        const bool has = !bad && p < task.nsel && k != 0;
        so.part_idx[row * DFLASH2_SHARD_LIST + p] = has ? static_cast<int32_t>(key_idx(k) + so.id_offset) : -1;
        so.part_z[row * DFLASH2_SHARD_LIST + p] = has ? key_val(k) : NEG_INF;
    }
    if (lane == 0) {
        so.part_m[row] = bad ? NAN : m;
        so.part_s[row] = bad ? NAN : (task.mode == MODE_TOPN_LSE && m != NEG_INF ? res.s : 0.0f);
    }
}

// Merge of S shard partials, one warp per row: the union of the lists as
// one list of keys (value, global id), the log normalisers combined, then
// the same outputs as the whole row's dflash2_topk16.
__global__ void __launch_bounds__(256) k_topk16_merge(int S, int64_t rows, const int32_t *part_idx,
                                                      const float *part_z, const float *part_m,
                                                      const float *part_s, int64_t V_total,
                                                      const dflash2_sampling *params, int64_t rows_per_param,
                                                      int32_t *cand_idx, float *cand_U, float *lse) {
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_wait();
    pdl_trigger();
    if (row >= rows) return;
    const RowTask task = decode_row(params, row / rows_per_param, V_total, false);
    RowResult<2> res;
    res.list.clear();
    res.best = 0;
    res.m = NEG_INF;
    res.s = 0.0f;
    res.bad = task.mode == MODE_SKIP;
    const float c = LOG2E / task.T;
    for (int sh = 0; sh < S; ++sh) {
        const int64_t base = (static_cast<int64_t>(sh) * rows + row) * DFLASH2_SHARD_LIST;
        WarpList<2> o;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int32_t id = part_idx[base + r * 32 + lane];
            o.k[r] = id >= 0 ? make_key(part_z[base + r * 32 + lane], static_cast<uint32_t>(id)) : 0ull;
        }
        res.list.merge(o, lane);  // each partial's list is already in key order
        const float m2 = part_m[static_cast<int64_t>(sh) * rows + row];
        const float s2 = part_s[static_cast<int64_t>(sh) * rows + row];
        if (m2 != m2) res.bad = true;
        else lse_combine(res.m, res.s, m2, s2, c);
    }
    if (task.mode == MODE_SKIP || task.mode == MODE_ARGMAX || task.wide) {
        if (lane < NC) {
            cand_idx[row * NC + lane] = -1;
            cand_U[row * NC + lane] = NAN;
        }
        if (lane == 0) lse[row] = NAN;
        return;
    }
    finalize_draft<2>(res, task, row, cand_idx, cand_U, lse, lane);
}

// Merge of S partials whose lists hold at most 16 entries (the fused LM
// head's, one per vocabulary range), one warp per row: each lane combines
// the log normalisers of shards lane, lane + 32, ... and the lanes combine in
// a fixed butterfly; the S * 16 candidate keys are loaded 256 at a time (all
// loads in flight at once) and sorted into the row's list 32 at a time.
__global__ void __launch_bounds__(256) k_topk16_merge16(int S, int64_t rows, const int32_t *part_idx,
                                                        const float *part_z, const float *part_m,
                                                        const float *part_s, int64_t V_total,
                                                        const dflash2_sampling *params, int64_t rows_per_param,
                                                        int32_t *cand_idx, float *cand_U, float *lse) {
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_wait();
    pdl_trigger();
    if (row >= rows) return;
    const RowTask task = decode_row(params, row / rows_per_param, V_total, false);
    const float c = LOG2E / task.T;
    float m = NEG_INF, sm = 0.0f;
    bool bad = task.mode == MODE_SKIP;
    for (int sh = lane; sh < S; sh += 32) {
        const float m2 = part_m[static_cast<int64_t>(sh) * rows + row];
        const float s2 = part_s[static_cast<int64_t>(sh) * rows + row];
        if (m2 != m2) bad = true;
        else lse_combine(m, sm, m2, s2, c);
    }
    bad = __any_sync(FULL, bad);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        const float m2 = __shfl_xor_sync(FULL, m, d);
        const float s2 = __shfl_xor_sync(FULL, sm, d);
        lse_combine(m, sm, m2, s2, c);
    }
    WarpList<1> acc;
    acc.clear();
    const int n = S * 16;
    for (int base = 0; base < n; base += 8 * 32) {
        uint64_t k[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = base + u * 32 + lane;
            const int64_t o = (static_cast<int64_t>(e >> 4) * rows + row) * DFLASH2_SHARD_LIST + (e & 15);
            const int32_t id = e < n ? part_idx[o] : -1;
            const float z = e < n ? part_z[o] : NEG_INF;
            k[u] = id >= 0 ? make_key(z, static_cast<uint32_t>(id)) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (!__any_sync(FULL, k[u] != 0)) continue;
            WarpList<1> o;
            o.k[0] = warp_sort_desc(k[u], lane);
            acc.merge(o, lane);
        }
    }
    if (task.mode == MODE_SKIP || task.mode == MODE_ARGMAX || task.nsel > 16) {
        if (lane < NC) {
            cand_idx[row * NC + lane] = -1;
            cand_U[row * NC + lane] = NAN;
        }
        if (lane == 0) lse[row] = NAN;
        return;
    }
    RowResult<1> res;
    res.list = acc;
    res.best = 0;
    res.m = m;
    res.s = sm;
    res.bad = bad;
    finalize_draft<1>(res, task, row, cand_idx, cand_U, lse, lane);
}

dflash2_status launch_merge16(int S, int64_t rows, const int32_t *part_idx, const float *part_z, const float *part_m,
                              const float *part_s, int64_t V_total, const dflash2_sampling *params,
                              int64_t rows_per_param, int32_t *cand_idx, float *cand_U, float *lse,
                              cudaStream_t stream) {
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffff) return DFLASH2_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_topk16_merge16, S, rows, part_idx, part_z, part_m, part_s, V_total, params,
                           rows_per_param, cand_idx, cand_U, lse) != cudaSuccess)
        return DFLASH2_ERR_CUDA;
    return after_launch();
}

// SAMPLED: some request may sample (params given): lists of 64 keys and every
// row mode; otherwise every row is greedy (top-16 and the log normaliser).
// Warps 0..SCAN_WARPS-1 stream the CTA's rows; the last warp completes each
// row (merges the warps' lists, joins the CTAs of a split row, writes outputs)
// while the others stream the next.
template <bool SAMPLED, bool BF16>
__global__ void __launch_bounds__(SCAN_THREADS, scan_min_blocks<SAMPLED>()) k_topk16(ScanGeom g, ScanWs sw,
                                                                                  int32_t *cand_idx,
                                                                                  float *cand_U, float *lse,
                                                                                  ShardOut so) {
    constexpr int R = SAMPLED ? 2 : 1;
    extern __shared__ unsigned char smem_raw[];
    ScanSmem &sm = *reinterpret_cast<ScanSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    // This grid reads its logits only after the grids before it completed;
    // from then on the next grid (the context gate reads nothing written
    // here) may start on the SMs this grid frees.
    scan_init(sm);
    pdl_wait();
    pdl_trigger();
    const int64_t begin = range_begin(g, blockIdx.x), end = range_begin(g, blockIdx.x + 1);
    const int64_t r_first = begin / g.cpr, r_last = (end - 1) / g.cpr;
    if (w < SCAN_WARPS) {
        WarpStream ws;
        stream_start(sm, g, ws, begin, end, w, lane, &g_err_topk);
        for (int64_t row = r_first; row <= r_last; ++row) {
            const int rrel = static_cast<int>(row - r_first);
            int w0;
            const int expect = row_warps(g, row, begin, end, &w0);
            const RowTask task = decode_row(g.params, row / g.rows_per_param, g.V_params, false);
            if (!SAMPLED || task.mode == MODE_TOPN_LSE)
                scan_row<R, MODE_TOPN_LSE, BF16>(sm, g, ws, task, row, rrel, expect, w0, false, &g_err_topk);
            else if (task.mode == MODE_TOPN)
                scan_row<R, MODE_TOPN, BF16>(sm, g, ws, task, row, rrel, expect, w0, false, &g_err_topk);
            else
                scan_row<R, MODE_ARGMAX, BF16>(sm, g, ws, task, row, rrel, expect, w0, true, &g_err_topk);
        }
        if (ws.aborted) stream_drain(sm, ws, w);
        if constexpr (!SAMPLED) return;  // greedy rows are never wide
    } else {
        bool aborted = false;
        uint32_t tail[SCAN_WARPS] = {0, 0, 0, 0};  // ring keys taken, per streaming warp
        for (int64_t row = r_first; row <= r_last; ++row) {
            const int rrel = static_cast<int>(row - r_first);
            const RowTask task = decode_row(g.params, row / g.rows_per_param, g.V_params, false);
            const float c = LOG2E / task.T;
            RowResult<R> res;
            bool done;
            if (!SAMPLED || task.mode == MODE_TOPN_LSE) {
                take_row<R, MODE_TOPN_LSE, BF16>(sm, g, row, res, rrel, c, task.nsel, tail, aborted, lane, &g_err_topk);
                done = join_parts<R, MODE_TOPN_LSE>(g, sw, row, res, c, lane);
            } else if (task.mode == MODE_TOPN) {
                take_row<R, MODE_TOPN, BF16>(sm, g, row, res, rrel, c, task.nsel, tail, aborted, lane, &g_err_topk);
                done = join_parts<R, MODE_TOPN>(g, sw, row, res, c, lane);
            } else {
                take_row<R, MODE_ARGMAX, BF16>(sm, g, row, res, rrel, c, task.nsel, tail, aborted, lane, &g_err_topk);
                if (blockIdx.x == range_owner(g, row * g.cpr)) {
                    if (so.part_idx) {
                        finalize_shard<R>(res, task, row, so, lane);
                    } else {
                        if (lane < NC) {
                            cand_idx[row * NC + lane] = -1;
                            cand_U[row * NC + lane] = NAN;
                        }
                        if (lane == 0) lse[row] = NAN;
                    }
                }
                continue;
            }
            if (done) {
                if (!res.bad) res.list = extract_topn<R, BF16>(g, row, res.list, task.nsel, sm.scratch, &sm.ngather, lane);
                if (so.part_idx) {
                    finalize_shard<R>(res, task, row, so, lane);
                } else if (task.wide) {
                    draft_wide_done<R, BF16>(sm, g, sw, res, task, row, cand_idx, cand_U, lse, lane);
                } else {
                    finalize_draft<R>(res, task, row, cand_idx, cand_U, lse, lane);
                }
            }
        }
    }
    if constexpr (SAMPLED) {
        __syncthreads();  // the stream buffers are idle from here
        if (sm.nwide > 0) draft_epilogue<BF16>(sm, g, sw, r_first, r_last, cand_U, lse);
    }
}

template <bool SAMPLED, bool BF16>
static dflash2_status launch_topk16(const ScanGeom &g, const ScanWs &sw, int32_t *cand_idx, float *cand_U,
                                    float *lse, const ShardOut &so, cudaStream_t stream) {
    const size_t smem = scan_smem_bytes();
    const void *fn = reinterpret_cast<const void *>(&k_topk16<SAMPLED, BF16>);
    const int64_t grid = scan_grid(blocks_per_sm(fn, SCAN_THREADS, smem), sm_count(), g.rows, g.total);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(SCAN_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_topk16<SAMPLED, BF16>, g, sw, cand_idx, cand_U, lse, so) != cudaSuccess)
        return DFLASH2_ERR_CUDA;
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

extern "C" size_t dflash2_topk16_workspace_bytes(int64_t rows) {
    if (rows < 0) return 0;
    return scan_ws_bytes(rows);
}

// Argument checks, then (with clear_tickets) zeroing of the rows' tickets in
// ws on `s`, then the launch.
static dflash2_status topk16_call(const void *logits, dflash2_dtype dt, int64_t rows, int64_t V, int64_t ld,
                                  const dflash2_sampling *params, int64_t rows_per_param, int32_t *cand_idx,
                                  float *cand_U, float *lse, void *ws, size_t ws_bytes, bool clear_tickets,
                                  cudaStream_t s, const ShardOut &so = ShardOut{}, int64_t V_params = 0) {
    if (!dtype_ok(dt) || rows < 0 || V < NC || V >= (int64_t(1) << 31) || ld < V || rows_per_param < 1)
        return DFLASH2_ERR_INVALID_ARG;
    const int es = esize(dt);
    if ((ld * es) % 16 != 0) return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!so.part_idx && (!cand_idx || !cand_U || !lse || !aligned16(cand_idx) || !aligned16(cand_U) || !aligned16(lse)))
        return DFLASH2_ERR_INVALID_ARG;
    if (!logits || !ws || !aligned16(logits) || !aligned16(ws) || (params && (reinterpret_cast<uintptr_t>(params) & 3)))
        return DFLASH2_ERR_INVALID_ARG;
    if (ws_bytes < scan_ws_bytes(rows)) return DFLASH2_ERR_WORKSPACE;
    ScanGeom g = make_geom(logits, ld, es, V, rows, params, rows_per_param);
    if (V_params > 0) g.V_params = V_params;
    const ScanWs sw = scan_ws_at(ws, rows);
    // the tickets and the wide marks, one range
    if (clear_tickets &&
        cudaMemsetAsync(sw.tickets, 0, scan_ws_rows_bytes(rows) + static_cast<size_t>(rows) * sizeof(int32_t), s) !=
            cudaSuccess)
        return DFLASH2_ERR_CUDA;
    if (params == nullptr)
        return dt == DFLASH2_BF16 ? launch_topk16<false, true>(g, sw, cand_idx, cand_U, lse, so, s)
                                  : launch_topk16<false, false>(g, sw, cand_idx, cand_U, lse, so, s);
    return dt == DFLASH2_BF16 ? launch_topk16<true, true>(g, sw, cand_idx, cand_U, lse, so, s)
                              : launch_topk16<true, false>(g, sw, cand_idx, cand_U, lse, so, s);
}

extern "C" dflash2_status dflash2_topk16(const void *logits, dflash2_dtype dt, int64_t rows, int64_t V,
                                         int64_t ld, const dflash2_sampling *params,
                                         int64_t rows_per_param, int32_t *cand_idx, float *cand_U,
                                         float *lse, void *ws, size_t ws_bytes, dflash2_stream stream) {
    return topk16_call(logits, dt, rows, V, ld, params, rows_per_param, cand_idx, cand_U, lse, ws, ws_bytes, false,
                       reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// dflash2_topk16_noalloc: the same call for callers that cannot hand this
// library any device memory of their own.  Its scratch -- one ticket per row
// and the partial records of rows split over several CTAs -- is a fixed array
// in the library's own device memory instead of a workspace.
namespace dfl {

constexpr int64_t TOPK_NOALLOC_MAX_ROWS = DFLASH2_TOPK16_NOALLOC_MAX_ROWS;
constexpr size_t TOPK_NOALLOC_BYTES = scan_ws_bytes(TOPK_NOALLOC_MAX_ROWS);

// Every GPU that loads the library holds this array (about 1.2 MB) until the
// process exits.  All calls share it.
static __device__ __align__(256) unsigned char g_topk_noalloc_ws[TOPK_NOALLOC_BYTES];

// Device address of the array on the current device, looked up once per
// device with that device current (in host code the array's name is only a
// host-side stand-in).  NULL if the lookup fails.
static void *topk_noalloc_ws() {
    static void *addr[64] = {nullptr};
    static std::mutex mu;
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_topk_noalloc_ws) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace dfl

extern "C" dflash2_status dflash2_topk16_noalloc(const void *logits, dflash2_dtype dt, int64_t rows, int64_t V,
                                                 int64_t ld, const dflash2_sampling *params, int64_t rows_per_param,
                                                 int32_t *cand_idx, float *cand_U, float *lse,
                                                 dflash2_stream stream) {
    if (rows > dfl::TOPK_NOALLOC_MAX_ROWS) return DFLASH2_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (rows <= 0)  // argument errors and the empty batch, reported as the workspace call does
        return topk16_call(logits, dt, rows, V, ld, params, rows_per_param, cand_idx, cand_U, lse, nullptr, 0,
                           false, s);
    void *ws = dfl::topk_noalloc_ws();
    if (!ws) return DFLASH2_ERR_CUDA;
    // The tickets and wide marks of the call's rows must start at zero.  A
    // call leaves them zero again, but one cut short (a launch error, or a
    // kernel that gave up on a bounded wait) may not, so every call clears
    // them first.  The partial records are written before they are read and
    // need no clearing.
    return topk16_call(logits, dt, rows, V, ld, params, rows_per_param, cand_idx, cand_U, lse, ws,
                       dfl::TOPK_NOALLOC_BYTES, true, s);
}

// ---------------------------------------------------------------------------
// Vocabulary-sharded top-16: each shard's partial, then the merge.
extern "C" dflash2_status dflash2_topk16_shard(const void *logits, dflash2_dtype dt, int64_t rows, int64_t V_shard,
                                               int64_t ld, int64_t id_offset, int64_t V_total,
                                               const dflash2_sampling *params, int64_t rows_per_param,
                                               int32_t *part_idx, float *part_z, float *part_m, float *part_s,
                                               void *ws, size_t ws_bytes, dflash2_stream stream) {
    if (id_offset < 0 || V_total < V_shard || id_offset + V_shard > V_total || V_total >= (int64_t(1) << 31))
        return DFLASH2_ERR_INVALID_ARG;
    if (rows > 0 && (!part_idx || !part_z || !part_m || !part_s || !aligned16(part_idx) || !aligned16(part_z) ||
                     (reinterpret_cast<uintptr_t>(part_m) & 3) || (reinterpret_cast<uintptr_t>(part_s) & 3)))
        return DFLASH2_ERR_INVALID_ARG;
    ShardOut so;
    so.part_idx = part_idx;
    so.part_z = part_z;
    so.part_m = part_m;
    so.part_s = part_s;
    so.id_offset = id_offset;
    if (rows > 0 && !part_idx) return DFLASH2_ERR_INVALID_ARG;
    return topk16_call(logits, dt, rows, V_shard, ld, params, rows_per_param, nullptr, nullptr, nullptr, ws,
                       ws_bytes, false, reinterpret_cast<cudaStream_t>(stream), so, V_total);
}

extern "C" dflash2_status dflash2_topk16_merge(int32_t S, int64_t rows, const int32_t *part_idx, const float *part_z,
                                               const float *part_m, const float *part_s, int64_t V_total,
                                               const dflash2_sampling *params, int64_t rows_per_param,
                                               int32_t *cand_idx, float *cand_U, float *lse, dflash2_stream stream) {
    if (S < 1 || S > DFLASH2_MAX_SHARDS || rows < 0 || V_total < NC || V_total >= (int64_t(1) << 31) ||
        rows_per_param < 1)
        return DFLASH2_ERR_INVALID_ARG;
    if (rows == 0) return DFLASH2_OK;
    if (!part_idx || !part_z || !part_m || !part_s || !cand_idx || !cand_U || !lse ||
        (params && (reinterpret_cast<uintptr_t>(params) & 3)))
        return DFLASH2_ERR_INVALID_ARG;
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffff) return DFLASH2_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_topk16_merge, static_cast<int>(S), rows, part_idx, part_z, part_m, part_s,
                           V_total, params, rows_per_param, cand_idx, cand_U, lse) != cudaSuccess)
        return DFLASH2_ERR_CUDA;
    return after_launch();
}
