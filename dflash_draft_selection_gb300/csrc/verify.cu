// verify.cu -- dflash2_verify: speculative-sampling verify of the proposed
// path against the target logits.
//
// FreeToken PR 857, "Details"/Sampled verify: accept a drafted token with
// probability min(1, p/q); on a reject resample from max(0, p - q), so the
// output follows the target distribution; all-greedy batches keep the prefix
// match.  DFlash 2 proposer issue, "Proposal" phase 3 (greedy stays
// longest-prefix; rejection sampling restores the exact target distribution).
// FreeToken PR 857, "Tests added or changed" (trusted, NaN, wrong-total and
// greedy rows) fixes the per-request error rows.
//
// One launch: persistent CTAs scan the B*(K+1) target rows (argmax for greedy
// requests, the filtered top-k distribution p for sampled ones) and publish a
// small record per row in the workspace; a per-request ticket lets the CTA
// that completes a request's last row run that request's accept walk.  For a
// sampled request each row's record also carries that position's decisions
// -- the checks of its q row, whether its drafted token is accepted, and the
// token a reject there (or, for the bonus row, the bonus) would emit -- taken
// when the row is finished, so that the accept walk reads them all at once
// and only picks the first reject.
#include "filter.cuh"
#include "host.hpp"
#include "rowscan.cuh"
#include "wide.cuh"

namespace dfl {

static __device__ unsigned int g_err_verify;

struct TRec {
    int32_t n;       // support size of p (1 for greedy rows)
    int32_t flags;   // DFLASH2_ST_* of the row
    // Sampled rows with flags == 0 (see row_decide): position t < K: qflag
    // (DFLASH2_ST_* of its q row and slot), accepted, and emit (the residual
    // draw when not accepted); the bonus row K: emit (the bonus draw).
    int32_t qflag;
    int32_t accepted;
    int32_t emit;
    int32_t ids[DFLASH2_MAX_TOPK];
    float p[DFLASH2_MAX_TOPK];
};

struct VerifyArgs {
    const int32_t *path_tok;
    const int32_t *cand_idx;
    const float *q_sel;
    const int32_t *path_slot;
    const float *u_acc;
    const float *u_res;
    uint32_t flags;
    int32_t *accept_len;
    int32_t *out_tok;
    int32_t *status;
    int32_t *tickets;
    TRec *recs;
    int K;
};

constexpr size_t TICKET_BYTES_ALIGN = 256;

// ---------------------------------------------------------------- records --
// The row's record.  For a sampled row also returns p's support as the
// accept walk reads it: entry i = r*32 + lane in (id[r], p[r]), -1 / 0 past
// the kept count *rn.  Returns the row's flags.
template <int R>
__device__ __forceinline__ int32_t finalize_target(const RowResult<R> &res, const RowTask &task, TRec *rec, int lane,
                                                   int32_t (&id)[2], float (&pr)[2], int *rn) {
    int32_t flags = DFLASH2_ST_OK;
    id[0] = id[1] = -1;
    pr[0] = pr[1] = 0.0f;
    *rn = 0;
    if (task.mode == MODE_ARGMAX) {
        const bool bad = res.bad || res.best == 0 || !isfinite(key_val(res.best));
        if (bad) flags = DFLASH2_ST_NAN;
        if (lane == 0) {
            rec->n = bad ? 0 : 1;
            rec->ids[0] = bad ? -1 : key_idx(res.best);
            rec->p[0] = 1.0f;
        }
    } else {
        const float z0 = key_val(res.list.k[0]);
        const float z0b = __shfl_sync(FULL, z0, 0);
        if (res.bad || !isfinite(z0b)) {
            flags = DFLASH2_ST_NAN;
            if (lane == 0) rec->n = 0;
        } else {
            float e[R], ek;
            const int kept = topn_filter<R>(res.list, task, z0b, lane, e, &ek);
            const float inv = 1.0f / ek;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int p = r * 32 + lane;
                if (p < kept) {
                    id[r] = key_idx(res.list.k[r]);
                    pr[r] = e[r] * inv;
                    rec->ids[p] = id[r];
                    rec->p[p] = pr[r];
                }
            }
            *rn = kept;
            if (lane == 0) rec->n = kept;
        }
    }
    if (lane == 0) rec->flags = flags;
    return flags;
}

// ------------------------------------------------------------ accept walk --
struct DrawScratch {
    int32_t ids[DFLASH2_MAX_TOPK];
    int32_t sid[DFLASH2_MAX_TOPK];
    float sw[DFLASH2_MAX_TOPK];
    double wr[NC];      // wide rows' draws: each candidate's r
    int32_t wcand[NC];  // and its id
};
static_assert(sizeof(DrawScratch) <= sizeof(ScanSmem::scratch), "the draw scratch fits the completion warp's scratch");
static_assert(sizeof(DrawScratch) <= sizeof(WideSmem::scratch), "the draw scratch fits the epilogue's scratch");

// Inverse CDF over the entries sorted by ascending token id: the first entry
// whose running weight exceeds u * (total weight); if rounding leaves none,
// the last entry with a positive weight.  Entries i < n are (id_i, w_i) with
// i = r*32 + lane; ids are distinct.  The entries are ranked by id in shared
// memory; then lane l holds sorted entries l and l + 32, and the running
// weights come from two warp scans.  Warp-uniform; returns the token.
__device__ int32_t draw_ascending(const int32_t (&id)[2], const float (&w)[2], int n, float u,
                                  DrawScratch &sc, int lane) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int i = r * 32 + lane;
        if (i < n) sc.ids[i] = id[r];
    }
    __syncwarp();
    int rank[2] = {0, 0};
    for (int j = 0; j < n; ++j) {
        const int32_t idj = sc.ids[j];
        rank[0] += idj < id[0];
        rank[1] += idj < id[1];
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int i = r * 32 + lane;
        if (i < n) {
            sc.sid[rank[r]] = id[r];
            sc.sw[rank[r]] = w[r];
        }
    }
    __syncwarp();
    const float w0 = lane < n ? sc.sw[lane] : 0.0f;
    const float w1 = lane + 32 < n ? sc.sw[lane + 32] : 0.0f;
    const float p0 = w0 > 0.0f ? w0 : 0.0f, p1 = w1 > 0.0f ? w1 : 0.0f;
    const float thr = u * warp_sum(p0 + p1);
    const float c0 = warp_inclusive_scan(p0, lane);
    const float c1 = warp_inclusive_scan(p1, lane) + __shfl_sync(FULL, c0, 31);
    const uint32_t h0 = __ballot_sync(FULL, w0 > 0.0f && c0 > thr);
    const uint32_t h1 = __ballot_sync(FULL, w1 > 0.0f && c1 > thr);
    const uint32_t l0 = __ballot_sync(FULL, w0 > 0.0f), l1 = __ballot_sync(FULL, w1 > 0.0f);
    int pos = -1;
    if (h0)
        pos = __ffs(h0) - 1;
    else if (h1)
        pos = 32 + __ffs(h1) - 1;
    else if (l1)
        pos = 32 + 31 - __clz(l1);
    else if (l0)
        pos = 31 - __clz(l0);
    const int32_t pick = pos >= 0 ? sc.sid[pos] : -1;
    __syncwarp();
    return pick;
}

__device__ __forceinline__ int32_t ldcg_i(const int32_t *p) { return __ldcg(p); }
__device__ __forceinline__ float ldcg_f(const float *p) { return __ldcg(p); }

// A sampled request's decisions at target row t of request b (rec), taken
// when the row is finished; (id, p, rn) is the row's p as finalize_target
// returns it.  Position t < K: the checks of its q row and slot (qflag: the
// first failing check, NaN or a negative q before a wrong total before a bad
// slot), whether u_acc * q < p at the drafted token, and -- when not -- the
// draw from max(0, p - q) (from p when that has no mass) with u_res[t].  The
// bonus row t = K: the draw from p with u_res[K].  The accept walk uses the
// decisions of the rows up to its first reject only.  Warp-uniform.
__device__ void row_decide(const VerifyArgs &a, int64_t b, int t, const int32_t (&id)[2], const float (&p)[2],
                           int rn, TRec *rec, DrawScratch &sc, int lane) {
    const int K = a.K;
    int32_t qflag = DFLASH2_ST_OK, accepted = 0, emit = -1;
    if (t < K) {
        const int64_t o = (b * K + t) * NC;
        const float qv = lane < NC ? a.q_sel[o + lane] : 0.0f;
        const int js = a.path_slot[b * K + t];
        const int32_t d = a.path_tok[b * K + t];
        if (__any_sync(FULL, lane < NC && (!isfinite(qv) || qv < 0.0f))) {
            qflag = DFLASH2_ST_NAN;
        } else {
            const float s = warp_sum(qv);
            if (!(a.flags & DFLASH2_VERIFY_TRUST_Q) && fabsf(s - 1.0f) > 1e-3f)
                qflag = DFLASH2_ST_BAD_Q;
            else if (js < 0 || js >= NC || a.cand_idx[o + js] != d)
                qflag = DFLASH2_ST_BAD_Q;
        }
        if (qflag == DFLASH2_ST_OK) {
            const float pd = warp_sum((id[0] == d && d >= 0 ? p[0] : 0.0f) + (id[1] == d && d >= 0 ? p[1] : 0.0f));
            const float qd = a.q_sel[o + js];
            accepted = a.u_acc[b * K + t] * qd < pd ? 1 : 0;
            if (!accepted) {
                // residual max(0, p - q) over the support of p
                const int32_t cc = lane < NC ? a.cand_idx[o + lane] : -1;
                float r_[2] = {0.0f, 0.0f};
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float qj_of = 0.0f;
                    for (int j = 0; j < NC; ++j) {
                        const int32_t cj = __shfl_sync(FULL, cc, j);
                        const float qj = __shfl_sync(FULL, qv, j);
                        if (cj == id[r]) qj_of = qj;
                    }
                    const float diff = p[r] - qj_of;
                    r_[r] = (r * 32 + lane < rn && diff > 0.0f) ? diff : 0.0f;
                }
                const float Z = warp_sum(r_[0] + r_[1]);
                const float u = a.u_res[b * (K + 1) + t];
                emit = Z > 1e-12f ? draw_ascending(id, r_, rn, u, sc, lane) : draw_ascending(id, p, rn, u, sc, lane);
            }
        }
    } else {
        emit = draw_ascending(id, p, rn, a.u_res[b * (K + 1) + K], sc, lane);
    }
    if (lane == 0) {
        rec->qflag = qflag;
        rec->accepted = accepted;
        rec->emit = emit;
    }
}

// The accept walk of request b (consumer warp 0 of the CTA that completed the
// request's rows).
template <bool SAMPLED>
__device__ void accept_request(const VerifyArgs &a, const dflash2_sampling *params, int64_t b,
                               int64_t V, DrawScratch &sc, int lane) {
    const int K = a.K;
    const RowTask rt = decode_row(params, b, V, true);
    const bool greedy = !SAMPLED || rt.mode == MODE_ARGMAX;
    const TRec *rec = a.recs + b * (K + 1);
    int st = DFLASH2_ST_OK;
    if (rt.mode == MODE_SKIP) {
        st = rt.status;
    } else {
        const int32_t fl = lane <= K ? ldcg_i(&rec[lane].flags) : DFLASH2_ST_OK;
        if (__any_sync(FULL, fl != DFLASH2_ST_OK)) st = DFLASH2_ST_NAN;
    }
    if (st == DFLASH2_ST_OK && greedy) {
        // All rows at once: lane t holds the target argmax of row t and the
        // drafted token of position t; the first mismatch ends the prefix.
        const int32_t g = lane <= K ? ldcg_i(&rec[lane].ids[0]) : -1;
        const int32_t d = lane < K ? a.path_tok[b * K + lane] : -1;
        const uint32_t miss = __ballot_sync(FULL, lane < K && d != g);
        const int n = miss ? __ffs(miss) - 1 : K;
        const int32_t emit = __shfl_sync(FULL, g, n);
        for (int i = lane; i <= K; i += 32) a.out_tok[b * (K + 1) + i] = i < n ? a.path_tok[b * K + i] : (i == n ? emit : -1);
        if (lane == 0) {
            a.accept_len[b] = n;
            a.status[b] = DFLASH2_ST_OK;
        }
        return;
    }
    int n = 0;
    int32_t emit = -1;
    if (st == DFLASH2_ST_OK) {
        // lane t <= K holds row t's decisions (row_decide); the first failing
        // q check decides the status, else the first reject ends the prefix
        const int32_t qf = lane < K ? ldcg_i(&rec[lane].qflag) : DFLASH2_ST_OK;
        const int32_t acc = lane < K ? ldcg_i(&rec[lane].accepted) : 1;
        const int32_t em = lane <= K ? ldcg_i(&rec[lane].emit) : -1;
        const uint32_t badq = __ballot_sync(FULL, qf != DFLASH2_ST_OK);
        if (badq) {
            st = __shfl_sync(FULL, qf, __ffs(badq) - 1);
        } else {
            const uint32_t rej = __ballot_sync(FULL, lane < K && acc == 0);
            n = rej ? __ffs(rej) - 1 : K;
            emit = __shfl_sync(FULL, em, n);
        }
    }
    for (int i = lane; i <= K; i += 32) {
        int32_t v = -1;
        if (st == DFLASH2_ST_OK) v = i < n ? a.path_tok[b * K + i] : (i == n ? emit : -1);
        a.out_tok[b * (K + 1) + i] = v;
    }
    if (lane == 0) {
        a.accept_len[b] = st == DFLASH2_ST_OK ? n : 0;
        a.status[b] = st;
    }
}

// ------------------------------------------------------ wide target rows --
// A sampled target row whose p reaches past its 64 best (top_p with top_k
// off, top_k above 64, or no filter at all): p(v) = w_v / P on the tokens
// the WideCut keeps, 0 elsewhere, with w_v = 2^((z_v - m) c) counted in the
// fixed point of the filter's passes.  The residual draw is an inverse CDF
// over ascending ids: block sums of the row (at most 255 blocks, one team
// pass that also counts each block's ties at the cut's value, so that the
// lowest-id ties are the kept ones), then the crossing block element by
// element.

// A wide row's state while it waits for the CTA's epilogue, kept in its
// record's support arrays (a wide row has no listed support).
struct WideStash {
    float m;        // the row maximum
    int32_t ready;  // the cut below is known (from the 64 best)
    int32_t cut;
    float P;
    uint32_t vk;
    int32_t all;
    int32_t nkeep;
    int32_t ties;   // -1: not known
};
static_assert(sizeof(WideStash) <= sizeof(int32_t) * DFLASH2_MAX_TOPK, "the stash fits a record's id array");

__device__ __forceinline__ void stash_put(TRec *rec, float m, bool ready, const WideCut &wc) {
    WideStash s;
    s.m = m;
    s.ready = ready ? 1 : 0;
    s.cut = static_cast<int32_t>(wc.cut);
    s.P = wc.P;
    s.vk = wc.vk;
    s.all = wc.all ? 1 : 0;
    s.nkeep = static_cast<int32_t>(wc.nkeep);
    s.ties = wc.ties == INT64_MAX ? -1 : static_cast<int32_t>(wc.ties);
    *reinterpret_cast<WideStash *>(rec->ids) = s;
}
__device__ __forceinline__ WideStash stash_get(const TRec *rec, WideCut *wc) {
    const WideStash s = *reinterpret_cast<const WideStash *>(rec->ids);
    wc->cut = s.cut;
    wc->P = s.P;
    wc->vk = s.vk;
    wc->all = s.all != 0;
    wc->nkeep = s.nkeep;
    wc->ties = s.ties < 0 ? INT64_MAX : s.ties;
    return s;
}

// The draw's blocks: nblk <= 255 of blk elements, blk a multiple of a
// warp's 32 vectors.
struct WideBlocks {
    int64_t blk;
    int nblk;
};
template <bool BF16>
__device__ __forceinline__ WideBlocks wide_blocks(int64_t V) {
    constexpr int SEG = 32 * VecLoad<BF16>::VE;
    int64_t blk = (V + 254) / 255;
    blk = (blk + SEG - 1) / SEG * SEG;
    return {blk, static_cast<int>((V + blk - 1) / blk)};
}

// One pass over the row: per block, the mass of the kept tokens relative to
// P (h.u.blk) and the ties at the cut's value in the blocks before it
// (h.cnt).  Team-wide; ends synchronised.
template <bool BF16>
__device__ void wide_block_pass(const Team &tm, WideSmem &sm, const ScanGeom &g, int64_t row, const WideCut &wc,
                                float m, float c, const Fx &fx, const WideBlocks &wb, int lane) {
    using VL = VecLoad<BF16>;
    constexpr int VE = VL::VE;
    constexpr int esz = BF16 ? 2 : 4;
    WideHist &h = sm.h;
    for (int i = tm.rank; i < 256; i += tm.size) {
        h.cnt[i] = 0;
        h.u.fx.lo[i] = 0;
        h.u.fx.hi[i] = 0;
    }
    tm.sync();
    const char *rowp = g.base + row * g.ld_bytes;
    const int64_t nvec = g.V * esz / 16;
    // a lane's elements: fixed-point mass above the cut's value, ties at it
    auto tally = [&](float x, bool valid, uint64_t &q, uint32_t &t) {
        if (!valid) return;
        const int s = wc.all ? 1 : (wide_vk<BF16>(x) > wc.vk ? 1 : (wide_vk<BF16>(x) == wc.vk ? 2 : 0));
        if (s == 1) q += wide_q(ex2((x - m) * c), fx);
        if (s == 2) ++t;
    };
    auto publish = [&](int64_t e0, uint64_t q, uint32_t t) {  // the warp's 32 vectors lie in one block
        const uint64_t qs = group_sum_q(FULL, q);
        const uint32_t ts = __reduce_add_sync(FULL, t);
        if (lane == 0 && (qs | ts)) {
            const int bi = static_cast<int>(e0 / wb.blk);
            fx_add(&h.u.fx.lo[bi], &h.u.fx.hi[bi], qs);
            atomicAdd(&h.cnt[bi], ts);
        }
    };
#pragma unroll 1
    for (int64_t v0 = tm.warp() * 32; v0 < nvec; v0 += 4 * static_cast<int64_t>(tm.size)) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t vi = v0 + u * tm.size + lane;
            v[u] = vi < nvec ? __ldcs(reinterpret_cast<const uint4 *>(rowp) + vi)
                             : make_uint4(VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD, VL::NEG_WORD);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t w0 = v0 + u * tm.size;  // the warp's first vector
            if (w0 >= nvec) break;                // warp-uniform
            float x[VE];
            VL::unpack(v[u], x);
            uint64_t q = 0;
            uint32_t t = 0;
#pragma unroll
            for (int e = 0; e < VE; ++e) tally(x[e], w0 + lane < nvec, q, t);
            publish(w0 * VE, q, t);
        }
    }
    if (tm.warp() == 0 && nvec * VE < g.V) {  // the ragged end (less than one vector)
        uint64_t q = 0;
        uint32_t t = 0;
        const int64_t i = nvec * VE + lane;
        tally(i < g.V ? VL::scalar(rowp, i) : NEG_INF, i < g.V, q, t);
        publish(nvec * VE, q, t);
    }
    tm.sync();
    // blocks 8 lane .. 8 lane + 7 of every warp: ties before each block, the
    // ties each keeps (the lowest ids first), its mass
    const uint64_t qcut = wc.all ? 0ull : wide_q(ex2((wide_vval<BF16>(wc.vk) - m) * c), fx);
    uint32_t tb[8], own = 0;
    double mb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int bi = lane * 8 + i;
        tb[i] = bi < wb.nblk ? h.cnt[bi] : 0u;
        own += tb[i];
    }
    uint32_t before = own;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL, before, d);
        if (lane >= d) before += t;
    }
    before -= own;
    const double invP = 1.0 / static_cast<double>(wc.P);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int bi = lane * 8 + i;
        int64_t kept = wc.nkeep - static_cast<int64_t>(before);
        kept = kept < 0 ? 0 : (kept > tb[i] ? tb[i] : kept);
        mb[i] = bi < wb.nblk ? static_cast<double>(fx_get(h, bi) + static_cast<uint64_t>(kept) * qcut) * fx.inv * invP
                             : 0.0;
        const uint32_t t = tb[i];
        tb[i] = before;
        before += t;
    }
    tm.sync();  // every warp read the sums before they are overwritten
    if (tm.warp() == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int bi = lane * 8 + i;
            if (bi < wb.nblk) {
                h.u.blk[bi] = mb[i];
                h.cnt[bi] = tb[i];
            }
        }
    }
    tm.sync();
}

// Rank by id among the ties at the cut's value of tie v: the ties of the
// blocks before v's, then those of v's block before v.  One thread; after
// the block pass.
template <bool BF16>
__device__ int64_t wide_tie_rank(const WideHist &h, const char *rowp, const WideCut &wc,
                                 const WideBlocks &wb, int64_t v) {
    const int64_t bi = v / wb.blk;
    int64_t r = h.cnt[bi];
    for (int64_t e = bi * wb.blk; e < v; ++e) r += wide_vk<BF16>(VecLoad<BF16>::scalar(rowp, e)) == wc.vk;
    return r;
}

// p(v) (0 outside the kept set or the vocabulary).  A tie at the cut's
// value needs the block pass first.  Per thread.
template <bool BF16>
__device__ double wide_p(const WideHist &h, const char *rowp, int64_t V, int32_t v, const WideCut &wc,
                         float m, float c, const Fx &fx, const WideBlocks &wb) {
    if (v < 0 || v >= V) return 0.0;
    const float z = VecLoad<BF16>::scalar(rowp, v);
    const int s = wide_side<BF16>(wc, z);
    if (s == 0) return 0.0;
    if (s == 2 && wide_tie_rank<BF16>(h, rowp, wc, wb, v) >= wc.nkeep) return 0.0;
    return static_cast<double>(wide_q(ex2((z - m) * c), fx)) * fx.inv / static_cast<double>(wc.P);
}

// Inverse CDF over ascending token ids of r (the residual max(0, p - q) with
// the candidates' q, or p itself for the bonus and when the residual has no
// mass): the first token whose running weight exceeds u * Z; if rounding
// leaves none, the last token with a positive weight.  After the block
// pass; every warp of the team computes the same token.
template <bool BF16>
__device__ int32_t wide_draw(const Team &tm, WideSmem &sm, DrawScratch &sc, const ScanGeom &g, int64_t row,
                             const WideCut &wc, float m, float c, const Fx &fx, const WideBlocks &wb,
                             int32_t cand, float qv, bool has_q, float u, int lane) {
    using VL = VecLoad<BF16>;
    const WideHist &h = sm.h;
    const char *rowp = g.base + row * g.ld_bytes;
    const int64_t V = g.V;
    // the candidates' p and r, and the residual's total Z = 1 - sum_j min(p_j, q_j)
    const double pj = has_q && lane < NC ? wide_p<BF16>(h, rowp, V, cand, wc, m, c, fx, wb) : 0.0;
    const double rj = has_q && lane < NC ? (pj > qv ? pj - qv : 0.0) : 0.0;
    double mn = has_q && lane < NC ? (pj < qv ? pj : static_cast<double>(qv)) : 0.0;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) mn += __shfl_xor_sync(FULL, mn, d);
    double Z = has_q ? 1.0 - mn : 1.0;
    bool use_cand = has_q;
    if (!(Z > 1e-12)) {  // no residual mass: draw from p
        Z = 1.0;
        use_cand = false;
    }
    if (tm.warp() == 0 && lane < NC) {
        sc.wcand[lane] = use_cand ? cand : -1;
        sc.wr[lane] = rj;
    }
    const double thr = static_cast<double>(u) * Z;
    // lane l holds blocks 8l .. 8l + 7; a candidate's block counts its r instead of its p
    double loc[8], ls = 0.0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int bi = lane * 8 + i;
        loc[i] = bi < wb.nblk ? h.u.blk[bi] : 0.0;
    }
    if (use_cand) {
        for (int j = 0; j < NC; ++j) {
            const int32_t cj = __shfl_sync(FULL, cand, j);
            const double dj = __shfl_sync(FULL, pj - rj, j);
            if (cj >= 0 && cj < V) {
                const int64_t bj = cj / wb.blk;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (lane * 8 + i == bj) loc[i] -= dj;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) ls += loc[i];
    tm.sync();  // the candidates' r in shared memory
    double before = ls;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const double t = __shfl_up_sync(FULL, before, d);
        if (lane >= d) before += t;
    }
    before -= ls;
    int hitb = -1, lastb = -1;
    double cb = before;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (loc[i] > 0.0) {
            if (hitb < 0 && cb + loc[i] > thr) hitb = lane * 8 + i;
            lastb = lane * 8 + i;
        }
        if (hitb < 0) cb += loc[i];
    }
    const uint32_t hm = __ballot_sync(FULL, hitb >= 0);
    const uint32_t lm = __ballot_sync(FULL, lastb >= 0);
    if (!hm && !lm) return -1;
    const bool fallback = hm == 0;
    const int src = fallback ? 31 - __clz(lm) : __ffs(hm) - 1;
    const int B = __shfl_sync(FULL, fallback ? lastb : hitb, src);
    const double cum0 = fallback ? -1.0 : __shfl_sync(FULL, cb, src);  // running weight before block B
    // within block B: lane l takes elements b0 + l * per .. + per - 1 in order
    const int64_t b0 = B * wb.blk, b1 = (b0 + wb.blk < V ? b0 + wb.blk : V);
    const int64_t per = wb.blk / 32;
    const int64_t s0 = b0 + lane * per, s1 = (s0 + per < b1 ? s0 + per : b1);
    const bool partial = !wc.all && wc.nkeep < wc.ties;
    // ties before this lane's elements
    uint32_t tl = 0;
    if (partial)
        for (int64_t e = s0; e < s1; ++e) tl += wide_vk<BF16>(VL::scalar(rowp, e)) == wc.vk;
    uint32_t tx = tl;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(FULL, tx, d);
        if (lane >= d) tx += t;
    }
    const int64_t rank0 = static_cast<int64_t>(h.cnt[B]) + (tx - tl);
    const double invP = 1.0 / static_cast<double>(wc.P);
    // r of element e of this lane, given the running tie rank
    auto r_of = [&](int64_t e, int64_t &rank) -> double {
        const float z = VL::scalar(rowp, e);
        int s = wc.all ? 1 : (wide_vk<BF16>(z) > wc.vk ? 1 : (wide_vk<BF16>(z) == wc.vk ? 2 : 0));
        if (s == 2) s = (!partial || rank < wc.nkeep) ? 1 : 0, ++rank;
        double r = s == 1 ? static_cast<double>(wide_q(ex2((z - m) * c), fx)) * fx.inv * invP : 0.0;
        if (use_cand) {
#pragma unroll 4
            for (int j = 0; j < NC; ++j)
                if (static_cast<int32_t>(e) == sc.wcand[j]) r = sc.wr[j];
        }
        return r;
    };
    double sub = 0.0;
    int64_t lastpos = -1;
    {
        int64_t rank = rank0;
        for (int64_t e = s0; e < s1; ++e) {
            const double r = r_of(e, rank);
            sub += r;
            if (r > 0.0) lastpos = e;
        }
    }
    double sb = sub;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const double t = __shfl_up_sync(FULL, sb, d);
        if (lane >= d) sb += t;
    }
    sb -= sub;
    const uint32_t pm = __ballot_sync(FULL, lastpos >= 0);
    const int32_t last_tok = pm ? static_cast<int32_t>(__shfl_sync(FULL, lastpos, 31 - __clz(pm))) : -1;
    if (fallback) return last_tok;
    const bool crosses = cum0 + sb + sub > thr && sub > 0.0;
    const uint32_t cm = __ballot_sync(FULL, crosses);
    if (!cm) return last_tok;  // rounding: the block's last positive token
    const int L = __ffs(cm) - 1;
    // lane L walks its elements in order
    int32_t pick = -1;
    if (lane == L) {
        double run = cum0 + sb;
        int64_t rank = rank0;
        for (int64_t e = s0; e < s1; ++e) {
            const double r = r_of(e, rank);
            if (r > 0.0) {
                run += r;
                if (run > thr) {
                    pick = static_cast<int32_t>(e);
                    break;
                }
            }
        }
        if (pick < 0) pick = static_cast<int32_t>(lastpos);  // rounding: the lane's last positive token
    }
    return __shfl_sync(FULL, pick, L);
}

// A wide sampled row's decisions at position t of request b (as row_decide
// takes them for rows whose p lies in their 64 best).  Team-wide; the
// record is written by the team's first thread.
template <bool BF16>
__device__ __forceinline__ void row_decide_wide(const Team &tm, WideSmem &sm, DrawScratch &sc, const ScanGeom &g,
                                const VerifyArgs &a, int64_t row, int64_t b, int t, const WideCut &wc, float m,
                                float c, TRec *rec, int lane) {
    const int K = a.K;
    const char *rowp = g.base + row * g.ld_bytes;
    const Fx fx = wide_fx(g.V);
    const WideBlocks wb = wide_blocks<BF16>(g.V);
    bool blocks = false;
    int32_t qflag = DFLASH2_ST_OK, accepted = 0, emit = -1;
    if (t < K) {
        const int64_t o = (b * K + t) * NC;
        const float qv = lane < NC ? a.q_sel[o + lane] : 0.0f;
        const int32_t cand = lane < NC ? a.cand_idx[o + lane] : -1;
        const int js = a.path_slot[b * K + t];
        const int32_t d = a.path_tok[b * K + t];
        if (__any_sync(FULL, lane < NC && (!isfinite(qv) || qv < 0.0f))) {
            qflag = DFLASH2_ST_NAN;
        } else {
            const float s = warp_sum(qv);
            if (!(a.flags & DFLASH2_VERIFY_TRUST_Q) && fabsf(s - 1.0f) > 1e-3f)
                qflag = DFLASH2_ST_BAD_Q;
            else if (js < 0 || js >= NC || a.cand_idx[o + js] != d)
                qflag = DFLASH2_ST_BAD_Q;
        }
        if (qflag == DFLASH2_ST_OK) {
            if (d >= 0 && d < g.V && wide_side<BF16>(wc, VecLoad<BF16>::scalar(rowp, d)) == 2) {
                wide_block_pass<BF16>(tm, sm, g, row, wc, m, c, fx, wb, lane);  // d's rank among the ties
                blocks = true;
            }
            const float pd = static_cast<float>(wide_p<BF16>(sm.h, rowp, g.V, d, wc, m, c, fx, wb));
            const float qd = a.q_sel[o + js];
            accepted = a.u_acc[b * K + t] * qd < pd ? 1 : 0;
            if (!accepted) {
                if (!blocks) wide_block_pass<BF16>(tm, sm, g, row, wc, m, c, fx, wb, lane);
                emit = wide_draw<BF16>(tm, sm, sc, g, row, wc, m, c, fx, wb, cand, qv, true,
                                       a.u_res[b * (K + 1) + t], lane);
            }
        }
    } else {
        wide_block_pass<BF16>(tm, sm, g, row, wc, m, c, fx, wb, lane);
        emit = wide_draw<BF16>(tm, sm, sc, g, row, wc, m, c, fx, wb, -1, 0.0f, false,
                               a.u_res[b * (K + 1) + K], lane);
    }
    if (tm.rank == 0) {
        rec->qflag = qflag;
        rec->accepted = accepted;
        rec->emit = emit;
    }
}

// Publish the row's record and, if it was the request's last row, run the
// accept walk.  Consumer warp 0.
template <bool SAMPLED>
__device__ void row_done(const VerifyArgs &a, const dflash2_sampling *params, int64_t row,
                         int64_t V, DrawScratch &sc, int lane) {
    const int64_t b = row / (a.K + 1);
    __syncwarp();
    int old = 0;
    if (lane == 0) old = atomic_add_acq_rel(&a.tickets[b], 1);
    old = __shfl_sync(FULL, old, 0);
    if (old == a.K) {
        if (lane == 0) a.tickets[b] = 0;  // zero again for the next call
        __syncwarp();
        accept_request<SAMPLED>(a, params, b, V, sc, lane);
    }
}

// A completed wide row: its record's flags; the cut from the list when it
// decides it; the rest (the passes and the decisions) is left to the CTA's
// epilogue, with the row's state stashed in its record and the row marked
// as this CTA's.  A bad row's record goes out now.
template <bool SAMPLED, int R, bool BF16>
__device__ __forceinline__ void target_wide_done(ScanSmem &sm, DrawScratch &sc, const ScanGeom &g, const ScanWs &sw,
                                                 const VerifyArgs &a, const RowResult<R> &res, const RowTask &task,
                                                 int64_t row, TRec *rec, int lane) {
    const bool bad = res.bad || !isfinite(res.m);
    if (lane == 0) {
        rec->n = 0;
        rec->flags = bad ? DFLASH2_ST_NAN : DFLASH2_ST_OK;
    }
    if constexpr (R == 2) {
        if (!bad) {
            WideCut wc;
            const bool ready =
                wide_cut_list<BF16>(res.list, res.m, res.s, LOG2E / task.T, task.ek, task.top_p, g.V, &wc, lane);
            if (lane == 0) {
                stash_put(rec, res.m, ready, wc);
                sw.marks[row] = static_cast<int32_t>(blockIdx.x) + 1;
                ++sm.nwide;
            }
            return;
        }
    }
    row_done<SAMPLED>(a, g.params, row, g.V, sc, lane);
}

// The rows this CTA marked, on all five warps once the CTA has streamed its
// range: the cut (unless the 64 best gave it), the row's decisions, then
// its record goes out (and the request's accept walk, if it was the last
// row).
template <bool BF16>
__device__ __forceinline__ void verify_epilogue(ScanSmem &ssm, const ScanGeom g, const ScanWs sw, const VerifyArgs a,
                                             int64_t r_first, int64_t r_last) {
    WideSmem &sm = wide_smem(ssm);
    DrawScratch &sc = *reinterpret_cast<DrawScratch *>(sm.scratch);
    const Team tm{static_cast<int>(threadIdx.x), SCAN_THREADS};
    const int lane = threadIdx.x & 31;
    const int32_t me = static_cast<int32_t>(blockIdx.x) + 1;
    for (int64_t row = r_first; row <= r_last; ++row) {
        if (sw.marks[row] != me) continue;  // the same for every thread: only this CTA writes `me`
        const RowTask task = decode_row(g.params, row / g.rows_per_param, g.V, true);
        const float cw = LOG2E / task.T;
        TRec *rec = a.recs + row;
        WideCut wc;
        const WideStash st = stash_get(rec, &wc);
        if (!st.ready) wc = wide_cut_passes<BF16>(tm, sm, g, row, st.m, cw, task.ek, task.top_p, lane);
        row_decide_wide<BF16>(tm, sm, sc, g, a, row, row / (a.K + 1), static_cast<int>(row % (a.K + 1)), wc, st.m,
                              cw, rec, lane);
        tm.sync();
        if (tm.warp() == 0) row_done<true>(a, g.params, row, g.V, sc, lane);
        tm.sync();
        if (threadIdx.x == 0) sw.marks[row] = 0;
    }
}

// SAMPLED: some request may sample (params given); otherwise every row is
// an argmax and every request greedy.  Warps 0..SCAN_WARPS-1 stream the
// CTA's rows; the last warp completes each row (joins the CTAs of a split
// row, writes its record and runs the accept walk of a completed request)
// while the others stream the next.
template <bool SAMPLED, bool BF16>
__global__ void __launch_bounds__(SCAN_THREADS, scan_min_blocks<SAMPLED, true>()) k_verify(ScanGeom g, ScanWs sw,
                                                                                  VerifyArgs a) {
    constexpr int R = SAMPLED ? 2 : 1;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    ScanSmem &sm = *reinterpret_cast<ScanSmem *>(base);
    DrawScratch &sc = *reinterpret_cast<DrawScratch *>(sm.scratch);
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    scan_init(sm);
    pdl_wait();  // nothing is read before the grids before this one completed
    pdl_trigger();  // the next grid waits for this one to complete before it reads anything
    const int64_t begin = range_begin(g, blockIdx.x), end = range_begin(g, blockIdx.x + 1);
    const int64_t r_first = begin / g.cpr, r_last = (end - 1) / g.cpr;
    if (w < SCAN_WARPS) {
        WarpStream ws;
        stream_start(sm, g, ws, begin, end, w, lane, &g_err_verify);
        for (int64_t row = r_first; row <= r_last; ++row) {
            const int rrel = static_cast<int>(row - r_first);
            int w0;
            const int expect = row_warps(g, row, begin, end, &w0);
            const RowTask task = decode_row(g.params, row / g.rows_per_param, g.V, true);
            if (!SAMPLED || task.mode == MODE_ARGMAX)
                scan_row<R, MODE_ARGMAX, BF16>(sm, g, ws, task, row, rrel, expect, w0, false, &g_err_verify);
            else if (task.mode == MODE_TOPN)
                scan_row<R, MODE_TOPN, BF16>(sm, g, ws, task, row, rrel, expect, w0, false, &g_err_verify);
            else if (task.mode == MODE_TOPN_LSE)
                scan_row<R, MODE_TOPN_LSE, BF16>(sm, g, ws, task, row, rrel, expect, w0, false, &g_err_verify);
            else
                scan_row<R, MODE_ARGMAX, BF16>(sm, g, ws, task, row, rrel, expect, w0, true, &g_err_verify);
        }
        if (ws.aborted) stream_drain(sm, ws, w);
        if constexpr (!SAMPLED) return;  // greedy rows are never wide
    } else {
        bool aborted = false;
        uint32_t tail[SCAN_WARPS] = {0, 0, 0, 0};  // ring keys taken, per streaming warp
        for (int64_t row = r_first; row <= r_last; ++row) {
            const int rrel = static_cast<int>(row - r_first);
            const RowTask task = decode_row(g.params, row / g.rows_per_param, g.V, true);
            TRec *rec = a.recs + row;
            RowResult<R> res;
            bool done;
            if (!SAMPLED || task.mode == MODE_ARGMAX) {
                take_row<R, MODE_ARGMAX, BF16>(sm, g, row, res, rrel, LOG2E, task.nsel, tail, aborted, lane, &g_err_verify);
                done = join_parts<R, MODE_ARGMAX>(g, sw, row, res, LOG2E, lane);
            } else if (task.mode == MODE_TOPN) {
                take_row<R, MODE_TOPN, BF16>(sm, g, row, res, rrel, LOG2E, task.nsel, tail, aborted, lane, &g_err_verify);
                done = join_parts<R, MODE_TOPN>(g, sw, row, res, LOG2E, lane);
                if (done && !res.bad) res.list = extract_topn<R, BF16>(g, row, res.list, task.nsel, sm.scratch, &sm.ngather, lane);
            } else if (task.mode == MODE_TOPN_LSE) {  // a wide row: the 64 best and the log normaliser
                const float cw = LOG2E / task.T;
                take_row<R, MODE_TOPN_LSE, BF16>(sm, g, row, res, rrel, cw, task.nsel, tail, aborted, lane, &g_err_verify);
                done = join_parts<R, MODE_TOPN_LSE>(g, sw, row, res, cw, lane);
                if (done && !res.bad) res.list = extract_topn<R, BF16>(g, row, res.list, task.nsel, sm.scratch, &sm.ngather, lane);
                if (done) target_wide_done<SAMPLED, R, BF16>(sm, sc, g, sw, a, res, task, row, rec, lane);
                continue;
            } else {
                take_row<R, MODE_ARGMAX, BF16>(sm, g, row, res, rrel, LOG2E, task.nsel, tail, aborted, lane, &g_err_verify);
                if (blockIdx.x == range_owner(g, row * g.cpr)) {
                    if (lane == 0) {
                        rec->n = 0;
                        rec->flags = task.status;
                    }
                    row_done<SAMPLED>(a, g.params, row, g.V, sc, lane);
                }
                continue;
            }
            if (done) {
                int32_t id[2];
                float pr[2];
                int rn;
                const int32_t fl = finalize_target<R>(res, task, rec, lane, id, pr, &rn);
                if (SAMPLED && task.mode == MODE_TOPN && fl == DFLASH2_ST_OK)
                    row_decide(a, row / (a.K + 1), static_cast<int>(row % (a.K + 1)), id, pr, rn, rec, sc, lane);
                row_done<SAMPLED>(a, g.params, row, g.V, sc, lane);
            }
        }
    }
    if constexpr (SAMPLED) {
        __syncthreads();  // the stream buffers are idle from here
        if (sm.nwide > 0) verify_epilogue<BF16>(sm, g, sw, a, r_first, r_last);
    }
}

template <bool SAMPLED, bool BF16>
static dflash2_status launch_verify(const ScanGeom &g, const ScanWs &sw, const VerifyArgs &a,
                                    cudaStream_t stream) {
    const size_t smem = scan_smem_bytes();
    const void *fn = reinterpret_cast<const void *>(&k_verify<SAMPLED, BF16>);
    const int64_t grid = scan_grid(blocks_per_sm(fn, SCAN_THREADS, smem), sm_count(), g.rows, g.total);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(SCAN_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_verify<SAMPLED, BF16>, g, sw, a) != cudaSuccess) return DFLASH2_ERR_CUDA;
    return after_launch();
}

unsigned int read_error_verify(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_err_verify, sizeof v);
    if (clear) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_err_verify, &z, sizeof z);
    }
    return v;
}

static size_t ticket_bytes(int64_t B) {
    return (static_cast<size_t>(B) * sizeof(int32_t) + TICKET_BYTES_ALIGN - 1) / TICKET_BYTES_ALIGN *
           TICKET_BYTES_ALIGN;
}

}  // namespace dfl

using namespace dfl;

static size_t recs_bytes(int64_t B, int32_t K) {
    return (static_cast<size_t>(B) * (K + 1) * sizeof(TRec) + 255) / 256 * 256;
}

extern "C" size_t dflash2_verify_workspace_bytes(int64_t B, int32_t K) {
    if (B < 0 || K < 1 || K > DFLASH2_MAX_K) return 0;
    return ticket_bytes(B) + recs_bytes(B, K) + scan_ws_bytes(B * (K + 1));
}

extern "C" dflash2_status dflash2_verify(const void *tlogits, dflash2_dtype dt, int64_t B, int32_t K,
                                         int64_t V, int64_t ld, const int32_t *path_tok,
                                         const int32_t *cand_idx, const float *q_sel,
                                         const int32_t *path_slot, const dflash2_sampling *params,
                                         const float *u_acc, const float *u_res, uint32_t flags,
                                         int32_t *accept_len, int32_t *out_tok, int32_t *status,
                                         void *ws, size_t ws_bytes, dflash2_stream stream) {
    if (!dtype_ok(dt) || B < 0 || K < 1 || K > DFLASH2_MAX_K || V < NC || V >= (int64_t(1) << 31) ||
        ld < V)
        return DFLASH2_ERR_INVALID_ARG;
    const int es = esize(dt);
    if ((ld * es) % 16 != 0) return DFLASH2_ERR_INVALID_ARG;
    if (B == 0) return DFLASH2_OK;
    if (!tlogits || !aligned16(tlogits) || !path_tok || !cand_idx || !q_sel || !path_slot ||
        !accept_len || !out_tok || !status || !ws)
        return DFLASH2_ERR_INVALID_ARG;
    if (params && (!u_acc || !u_res)) return DFLASH2_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 15) != 0) return DFLASH2_ERR_INVALID_ARG;
    if (ws_bytes < dflash2_verify_workspace_bytes(B, K)) return DFLASH2_ERR_WORKSPACE;
    const ScanGeom g = make_geom(tlogits, ld, es, V, B * (K + 1), params, K + 1);
    const ScanWs sw = scan_ws_at(static_cast<char *>(ws) + ticket_bytes(B) + recs_bytes(B, K), B * (K + 1));
    VerifyArgs a;
    a.path_tok = path_tok;
    a.cand_idx = cand_idx;
    a.q_sel = q_sel;
    a.path_slot = path_slot;
    a.u_acc = u_acc;
    a.u_res = u_res;
    a.flags = flags;
    a.accept_len = accept_len;
    a.out_tok = out_tok;
    a.status = status;
    a.tickets = static_cast<int32_t *>(ws);
    a.recs = reinterpret_cast<TRec *>(static_cast<char *>(ws) + ticket_bytes(B));
    a.K = K;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (params == nullptr)
        return dt == DFLASH2_BF16 ? launch_verify<false, true>(g, sw, a, s)
                                  : launch_verify<false, false>(g, sw, a, s);
    return dt == DFLASH2_BF16 ? launch_verify<true, true>(g, sw, a, s) : launch_verify<true, false>(g, sw, a, s);
}
