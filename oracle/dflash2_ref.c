/*
 * dflash2_ref.c -- CPU oracle for the DFlash 2 draft-selection + verify path.
 *
 * TEST INFRASTRUCTURE.  This file is a plain, slow restatement of what the
 * method computes, in fp64, written from the DFlash 2 pages:
 *   - "qwen3/dflash: DFlash 2 proposer -- top-16 path selector + two-tap
 *     dynamic convolution" (pegainfer issue 930), section "What upstream
 *     shipped" items 1-2 and "Proposal" phases 1-3;
 *   - FreeToken PR 857 "DFlash 2 next to MTP", section "Details" (Runtime,
 *     Sampled verify, Refused at startup) and "Tests added or changed".
 * Only tests, the smoke check and the bench's CPU-baseline leg may load it.
 * It shares no code, header or table with the CUDA library.
 *
 * Conventions
 *   - bf16 is widened to f32 by a 16-bit shift (exact); all sums are fp64.
 *   - Order key: token x ranks before y iff z_x > z_y, or z_x == z_y and
 *     x < y (lower token id wins ties).
 *   - Sampling parameters per request: temperature T (0 = greedy), top_k
 *     (0 = off), top_p (1 = off).  Filters apply in the order temperature ->
 *     top_k -> renormalise -> top_p -> renormalise.
 *
 * Parity pins: every function here is pinned by a test that does not use the
 * function itself (closed forms, brute force, library sorts, Monte Carlo);
 * the absolute values of the selector scores have no printed worked example
 * on the pages ("parity unpinned" against the pages for those values; they are
 * pinned to a direct triple-loop restatement and to the A=0 reduction).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define REF_F32 0
#define REF_BF16 1
#define NC 16 /* candidates per draft position */

/* per-request status codes */
#define REF_ST_OK 0
#define REF_ST_NAN 1
#define REF_ST_BAD_Q 2
#define REF_ST_BAD_PARAMS 3

static double ref_load(const void *p, int dtype, int64_t i) {
    if (dtype == REF_BF16) {
        uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    return (double)((const float *)p)[i];
}

typedef struct {
    double v;
    int32_t id;
} entry;

/* qsort comparator: larger value first, then lower token id. */
static int entry_cmp(const void *pa, const void *pb) {
    const entry *a = (const entry *)pa, *b = (const entry *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

static int id_cmp(const void *pa, const void *pb) {
    const entry *a = (const entry *)pa, *b = (const entry *)pb;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

/* A row is unusable when it holds a NaN or +Inf, or no finite-or-above value
 * at all (every logit -Inf).  -Inf alone is a masked token and is allowed. */
static int row_is_bad(const void *row, int dtype, int64_t V) {
    int any_above_minus_inf = 0;
    for (int64_t v = 0; v < V; v++) {
        double z = ref_load(row, dtype, v);
        if (isnan(z) || (isinf(z) && z > 0)) return 1;
        if (!(isinf(z) && z < 0)) any_above_minus_inf = 1;
    }
    return !any_above_minus_inf;
}

static int params_bad(double T, int32_t top_k, double top_p) {
    if (!(T >= 0.0) || isinf(T)) return 1;
    if (top_k < 0) return 1;
    if (!(top_p > 0.0 && top_p <= 1.0)) return 1;
    return 0;
}

/* Sort the whole row by the order key (a library sort serves as the step
 * "keep the candidates in rank order").  Caller frees. */
static entry *sorted_row(const void *row, int dtype, int64_t V) {
    entry *e = (entry *)malloc((size_t)V * sizeof(entry));
    for (int64_t v = 0; v < V; v++) {
        double z = ref_load(row, dtype, v);
        if (z == 0.0) z = 0.0; /* -0 and +0 are the same value: the id decides */
        e[v].v = z;
        e[v].id = (int32_t)v;
    }
    qsort(e, (size_t)V, sizeof(entry), entry_cmp);
    return e;
}

/*
 * Sampling filter on a sorted row (T > 0): temperature, then keep the first
 * top_k tokens and renormalise, then keep the shortest prefix whose
 * cumulative mass reaches top_p and renormalise.  Returns the number of kept
 * tokens; prob[i] is the final probability of ord[i] for i < kept.  *logZ is
 * the log normaliser of the kept set on the z/T scale, so that
 * log prob[i] = ord[i].v / T - *logZ.  *margin receives the smallest distance
 * between a cumulative mass and top_p seen while deciding the prefix (inf
 * when top_p is off).
 * FreeToken PR 857 "Speed" (temperature=1.0, top_p=0.95, top_k=20 on both
 * sides); the order of the filters is the usual one (a reading: the pages do
 * not state it).
 */
static int64_t ref_filter(const entry *ord, int64_t V, double T, int32_t top_k, double top_p,
                          double *prob, double *logZ, double *margin) {
    int64_t k = (top_k == 0 || top_k >= V) ? V : top_k;
    double M = ord[0].v / T;
    double Ek = 0.0;
    for (int64_t i = 0; i < k; i++) Ek += exp(ord[i].v / T - M);
    int64_t kept = k;
    *margin = INFINITY;
    if (top_p < 1.0) {
        double cum = 0.0;
        for (int64_t i = 0; i < k; i++) {
            cum += exp(ord[i].v / T - M) / Ek;
            double d = fabs(cum - top_p);
            if (d < *margin) *margin = d;
            if (cum >= top_p) {
                kept = i + 1;
                break;
            }
        }
    }
    double Ekept = 0.0;
    for (int64_t i = 0; i < kept; i++) Ekept += exp(ord[i].v / T - M);
    for (int64_t i = 0; i < kept; i++) prob[i] = exp(ord[i].v / T - M) / Ekept;
    *logZ = M + log(Ekept);
    return kept;
}

/* ------------------------------------------------------------------------ */
/* (1) top-16 candidates per draft position and their log-probabilities U.  */
/* ------------------------------------------------------------------------ */
/*
 * DFlash 2 proposer issue, "What upstream shipped" item 1 ("keep top-16
 * candidates per position"); FreeToken PR 857 "Details"/Runtime (the LM head
 * gives 16 candidates per slot).  U is the drafter's log-softmax at the
 * candidate (a reading: the pages leave U unspecified); greedy rows use
 * temperature 1; filtered rows use the log of the filtered distribution and
 * -inf for a candidate the filter drops.  lse is the log normaliser of the
 * distribution U is taken from, on the z/T' scale.
 * margin[r] (optional) = top_p decision margin of the row (inf if none).
 * Unusable rows and invalid parameters give idx -1, U NaN, lse NaN.
 */
/* The outputs of (1) for one usable row whose V entries are sorted by the
 * order key: idx/U are the row's 16 slots, *lse its normaliser, *margin its
 * top_p decision margin (inf when none). */
static void topk16_sorted(const entry *ord, int64_t V, double T, int32_t tk, double tp, int32_t *idx, double *U,
                          double *lse, double *margin) {
    for (int j = 0; j < NC; j++) idx[j] = ord[j].id;
    int filtered = T > 0.0 && ((tk > 0 && tk < V) || tp < 1.0);
    *margin = INFINITY;
    if (!filtered) {
        double Tp = T > 0.0 ? T : 1.0;
        double M = ord[0].v / Tp, S = 0.0;
        for (int64_t i = 0; i < V; i++) S += exp(ord[i].v / Tp - M);
        double L = M + log(S);
        *lse = L;
        for (int j = 0; j < NC; j++) U[j] = ord[j].v / Tp - L;
    } else {
        double *prob = (double *)malloc((size_t)V * sizeof(double));
        double L, mg;
        int64_t kept = ref_filter(ord, V, T, tk, tp, prob, &L, &mg);
        *lse = L;
        *margin = mg;
        for (int j = 0; j < NC; j++) U[j] = (j < kept) ? ord[j].v / T - L : -INFINITY;
        free(prob);
    }
}

void dflash2_ref_topk16(const void *logits, int dtype, int64_t rows, int64_t V, int64_t ld,
                        const float *temperature, const int32_t *top_k, const float *top_p,
                        int64_t rows_per_param, int32_t *cand_idx, double *cand_U, double *lse,
                        double *margin) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; r++) {
        const void *row = (const char *)logits + (size_t)(r * ld) * (dtype == REF_BF16 ? 2 : 4);
        int64_t pi = rows_per_param > 0 ? r / rows_per_param : 0;
        double T = temperature ? temperature[pi] : 0.0;
        int32_t tk = top_k ? top_k[pi] : 0;
        double tp = top_p ? top_p[pi] : 1.0;
        if (margin) margin[r] = INFINITY;
        if (params_bad(T, tk, tp) || row_is_bad(row, dtype, V)) {
            for (int j = 0; j < NC; j++) {
                cand_idx[r * NC + j] = -1;
                cand_U[r * NC + j] = NAN;
            }
            lse[r] = NAN;
            continue;
        }
        entry *ord = sorted_row(row, dtype, V);
        double mg;
        topk16_sorted(ord, V, T, tk, tp, cand_idx + r * NC, cand_U + r * NC, lse + r, &mg);
        if (margin) margin[r] = mg;
        free(ord);
    }
}

/* ------------------------------------------------------------------------ */
/* (1b) top-16 over a vocabulary split into shards: partials and merge.      */
/* ------------------------------------------------------------------------ */
/*
 * A tensor-parallel LM head leaves each GPU the logits of one slice of the
 * vocabulary.  The candidates and U of the whole row follow from one small
 * partial per slice, exchanged once (a reading of this library: the pages
 * run the drafter on one GPU with --tp 1).  Both functions restate the
 * definitions of (1) over the union of the slices.
 *
 * Row length of a partial's list for parameters (T, top_k, top_p) and the
 * whole vocabulary V_total: 16 for greedy and unfiltered rows, max(16, top_k)
 * for rows filtered with 0 < top_k < V_total; rows whose filter needs more
 * than P tokens (top_p < 1 with top_k off, or top_k > P) need the whole row
 * and are not supported: their partials and merged outputs are -1 / NaN.
 */
static int shard_list_len(double T, int32_t tk, double tp, int64_t V_total, int P) {
    if (T == 0.0) return NC;
    int filtered = (tk > 0 && tk < V_total) || tp < 1.0;
    if (!filtered) return NC;
    if (tk == 0 || tk >= V_total || tk > P) return -1; /* needs the whole row */
    return tk > NC ? tk : NC;
}

/*
 * Partial of the shard holding tokens [off, off + Vs) of each row:
 *   part_idx[r, i], part_z[r, i] (i < P): the shard's i-th token in the order
 *     key, as a global id (off + v) and its logit, for i below the row's
 *     list length (and below Vs); -1 and -inf after.
 *   part_m[r]: the shard's largest logit; part_s[r]: the sum over the shard of
 *     exp((z - part_m) / T'), T' = T for sampled rows and 1 for greedy rows;
 *     0 for filtered rows (their merge uses the lists alone).
 *   A shard row holding a NaN or +Inf, a row with invalid parameters and an
 *   unsupported row: idx -1, m NaN, s NaN.  A shard row whose logits are all
 *   -Inf is a slice of masked tokens: its list holds them (value -inf),
 *   m = -inf, s = 0.
 */
void dflash2_ref_topk16_shard(const void *logits, int dtype, int64_t rows, int64_t Vs, int64_t ld,
                              int64_t off, int64_t V_total, const float *temperature,
                              const int32_t *top_k, const float *top_p, int64_t rows_per_param, int P,
                              int32_t *part_idx, double *part_z, double *part_m, double *part_s) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; r++) {
        const void *row = (const char *)logits + (size_t)(r * ld) * (dtype == REF_BF16 ? 2 : 4);
        int64_t pi = rows_per_param > 0 ? r / rows_per_param : 0;
        double T = temperature ? temperature[pi] : 0.0;
        int32_t tk = top_k ? top_k[pi] : 0;
        double tp = top_p ? top_p[pi] : 1.0;
        for (int i = 0; i < P; i++) {
            part_idx[r * P + i] = -1;
            part_z[r * P + i] = -INFINITY;
        }
        int n = params_bad(T, tk, tp) ? -1 : shard_list_len(T, tk, tp, V_total, P);
        int bad = n < 0;
        for (int64_t v = 0; v < Vs && !bad; v++) {
            double z = ref_load(row, dtype, v);
            if (isnan(z) || (isinf(z) && z > 0)) bad = 1;
        }
        if (bad) {
            part_m[r] = NAN;
            part_s[r] = NAN;
            continue;
        }
        entry *ord = sorted_row(row, dtype, Vs);
        for (int i = 0; i < n && i < Vs; i++) {
            part_idx[r * P + i] = (int32_t)(off + ord[i].id);
            part_z[r * P + i] = ord[i].v;
        }
        double m = ord[0].v;
        part_m[r] = m;
        int filtered = T > 0.0 && ((tk > 0 && tk < V_total) || tp < 1.0);
        double S = 0.0;
        if (!filtered && !isinf(m)) {
            double Tp = T > 0.0 ? T : 1.0;
            for (int64_t i = 0; i < Vs; i++) S += exp((ord[i].v - m) / Tp);
        }
        part_s[r] = S;
        free(ord);
    }
}

/*
 * Merge of S partials (part_* laid out [S, rows, P] and [S, rows]) into the
 * row's cand_idx [rows, 16], cand_U and lse as (1) defines them for the whole
 * row of V_total tokens: the union of the lists in the order key; for
 * unfiltered rows lse = log sum_s exp(m_s / T') s_s (its largest term
 * factored out) and U = z / T' - lse; for filtered rows the filter of (1) on
 * the sorted union.  A row with a NaN partial, or none with a finite
 * largest logit, and an unsupported row get -1 / NaN.
 */
void dflash2_ref_topk16_merge(int S, int64_t rows, int P, const int32_t *part_idx, const double *part_z,
                              const double *part_m, const double *part_s, int64_t V_total,
                              const float *temperature, const int32_t *top_k, const float *top_p,
                              int64_t rows_per_param, int32_t *cand_idx, double *cand_U, double *lse,
                              double *margin) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; r++) {
        int64_t pi = rows_per_param > 0 ? r / rows_per_param : 0;
        double T = temperature ? temperature[pi] : 0.0;
        int32_t tk = top_k ? top_k[pi] : 0;
        double tp = top_p ? top_p[pi] : 1.0;
        if (margin) margin[r] = INFINITY;
        int bad = params_bad(T, tk, tp) || shard_list_len(T, tk, tp, V_total, P) < 0;
        double M = -INFINITY;
        for (int s = 0; s < S && !bad; s++) {
            double m = part_m[(int64_t)s * rows + r];
            if (isnan(m)) bad = 1;
            else if (m > M) M = m;
        }
        if (!bad && !isfinite(M)) bad = 1;
        if (bad) {
            for (int j = 0; j < NC; j++) {
                cand_idx[r * NC + j] = -1;
                cand_U[r * NC + j] = NAN;
            }
            lse[r] = NAN;
            continue;
        }
        entry *u = (entry *)malloc((size_t)S * P * sizeof(entry));
        int64_t n = 0;
        for (int s = 0; s < S; s++)
            for (int i = 0; i < P; i++) {
                int64_t k = ((int64_t)s * rows + r) * P + i;
                if (part_idx[k] < 0) continue;
                u[n].v = part_z[k] == 0.0 ? 0.0 : part_z[k];
                u[n].id = part_idx[k];
                n++;
            }
        qsort(u, (size_t)n, sizeof(entry), entry_cmp);
        for (int j = 0; j < NC; j++) cand_idx[r * NC + j] = j < n ? u[j].id : -1;
        int filtered = T > 0.0 && ((tk > 0 && tk < V_total) || tp < 1.0);
        if (!filtered) {
            double Tp = T > 0.0 ? T : 1.0, sum = 0.0;
            for (int s = 0; s < S; s++) {
                double m = part_m[(int64_t)s * rows + r];
                if (!isinf(m)) sum += part_s[(int64_t)s * rows + r] * exp((m - M) / Tp);
            }
            double L = M / Tp + log(sum);
            lse[r] = L;
            for (int j = 0; j < NC; j++) cand_U[r * NC + j] = j < n ? u[j].v / Tp - L : -INFINITY;
        } else {
            double *prob = (double *)malloc((size_t)n * sizeof(double));
            double L, mg;
            int64_t kept = ref_filter(u, n, T, tk, tp, prob, &L, &mg);
            lse[r] = L;
            if (margin) margin[r] = mg;
            for (int j = 0; j < NC; j++) cand_U[r * NC + j] = (j < kept) ? u[j].v / T - L : -INFINITY;
            free(prob);
        }
        free(u);
    }
}

/* ------------------------------------------------------------------------ */
/* (1c) the LM head and the top-16 in one: z = h . W^T, then (1).            */
/* ------------------------------------------------------------------------ */
/*
 * DFlash 2 proposer issue, "What upstream shipped" item 1 and FreeToken PR
 * 857 "Details"/Runtime (the candidates come from the LM head): the logits
 * of row r are z_v = sum_k h[r,k] W[v,k] (bf16 inputs, exact fp64 products
 * and sums), and the outputs are those of (1) on them.  Rows that would need
 * more than 16 candidates (a top_k filter above 16) or the whole row (top_p
 * with top_k off) get -1 / NaN, as the library's fused kernel gives them.
 * gap[r] (optional): the smallest difference between consecutive logits
 * among the row's 17 best, the margin of the candidates' order.
 */
void dflash2_ref_lmhead_topk16(const void *h, const void *W, int dtype, int64_t rows, int64_t hidden, int64_t V,
                               const float *temperature, const int32_t *top_k, const float *top_p,
                               int64_t rows_per_param, int32_t *cand_idx, double *cand_U, double *lse,
                               double *margin, double *gap) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; r++) {
        int64_t pi = rows_per_param > 0 ? r / rows_per_param : 0;
        double T = temperature ? temperature[pi] : 0.0;
        int32_t tk = top_k ? top_k[pi] : 0;
        double tp = top_p ? top_p[pi] : 1.0;
        if (margin) margin[r] = INFINITY;
        if (gap) gap[r] = INFINITY;
        int need = T == 0.0 || !((tk > 0 && tk < V) || tp < 1.0) ? NC : ((tk == 0 || tk >= V) ? -1 : tk);
        entry *ord = (entry *)malloc((size_t)V * sizeof(entry));
        int bad = params_bad(T, tk, tp) || need < 0 || need > NC;
        for (int64_t v = 0; v < V && !bad; v++) {
            double z = 0.0;
            for (int64_t k = 0; k < hidden; k++) z += ref_load(h, dtype, r * hidden + k) * ref_load(W, dtype, v * hidden + k);
            if (isnan(z) || isinf(z)) bad = 1;
            ord[v].v = z == 0.0 ? 0.0 : z;
            ord[v].id = (int32_t)v;
        }
        if (bad) {
            for (int j = 0; j < NC; j++) {
                cand_idx[r * NC + j] = -1;
                cand_U[r * NC + j] = NAN;
            }
            lse[r] = NAN;
            free(ord);
            continue;
        }
        qsort(ord, (size_t)V, sizeof(entry), entry_cmp);
        double mg;
        topk16_sorted(ord, V, T, tk, tp, cand_idx + r * NC, cand_U + r * NC, lse + r, &mg);
        if (margin) margin[r] = mg;
        if (gap)
            for (int j = 0; j < NC && j + 1 < V; j++)
                if (ord[j].v - ord[j + 1].v < gap[r]) gap[r] = ord[j].v - ord[j + 1].v;
        free(ord);
    }
}

/* ------------------------------------------------------------------------ */
/* (2) context gate H(h) = sigmoid(W_g h).                                   */
/* ------------------------------------------------------------------------ */
/* DFlash 2 proposer issue, "What upstream shipped" item 1 (context gate of
 * the low-rank bilinear attention); the form sigmoid(W_g h) with W_g of shape
 * [D, hidden] and no bias is the reading this library takes. */
void dflash2_ref_ctx_gate(const void *h, int dtype, int64_t n, int64_t hidden, const void *Wg,
                          int64_t D, double *gate) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        for (int64_t k = 0; k < D; k++) {
            double acc = 0.0;
            for (int64_t c = 0; c < hidden; c++)
                acc += ref_load(Wg, dtype, k * hidden + c) * ref_load(h, dtype, i * hidden + c);
            gate[i * D + k] = 1.0 / (1.0 + exp(-acc));
        }
    }
}

/* ------------------------------------------------------------------------ */
/* (3) pairwise scores S_t(a,b) = U_t(b) + <A(a) * H(h_t), B(b)>.            */
/* ------------------------------------------------------------------------ */
/*
 * DFlash 2 proposer issue, "What upstream shipped" item 1 and "Proposal"
 * phase 1 (block_size x 16 preds x 16 cands x 256 dims).  scores is
 * [B, K, 16, 16]: scores[b,t,i,j] pairs predecessor i with candidate j of
 * position t.  At t = 0 the only predecessor is the last verified token
 * (row 0); rows 1..15 are -inf.  For t >= 1 the predecessors are the
 * candidates of position t-1.  A candidate or predecessor id outside [0, V)
 * gives NaN scores in its column or row.
 */
void dflash2_ref_pair_scores(int64_t B, int K, const int32_t *cand_idx, const double *cand_U,
                             const int32_t *last_tok, const void *A, const void *Bt, int dtype,
                             int64_t V, int D, const double *gate, double *scores) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; b++) {
        for (int t = 0; t < K; t++) {
            const int32_t *cand = cand_idx + (b * K + t) * NC;
            const double *U = cand_U + (b * K + t) * NC;
            const double *g = gate + (b * K + t) * D;
            double *S = scores + (b * K + t) * NC * NC;
            for (int i = 0; i < NC; i++) {
                int has_pred = (t > 0) || (i == 0);
                int32_t a = (t == 0) ? last_tok[b] : cand_idx[(b * K + t - 1) * NC + i];
                for (int j = 0; j < NC; j++) {
                    if (!has_pred) {
                        S[i * NC + j] = -INFINITY;
                        continue;
                    }
                    int32_t c = cand[j];
                    if (a < 0 || a >= V || c < 0 || c >= V) {
                        S[i * NC + j] = NAN;
                        continue;
                    }
                    double dot = 0.0;
                    for (int k = 0; k < D; k++)
                        dot += ref_load(A, dtype, (int64_t)a * D + k) * g[k] *
                               ref_load(Bt, dtype, (int64_t)c * D + k);
                    S[i * NC + j] = U[j] + dot;
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* (4) the walk over the precomputed scores.                                 */
/* ------------------------------------------------------------------------ */
/*
 * DFlash 2 proposer issue, "What upstream shipped" item 1 ("a single
 * greedy/sampled walk over the precomputed scores picks the proposed path")
 * and "Proposal" phase 1 (a <= block_size-step argmax walk); FreeToken PR 857
 * "Details"/Runtime (sampled from its distribution q, or argmax when greedy).
 * Step t looks at the score row of the previously chosen slot (row 0 at
 * t = 0).  Greedy: the first slot holding the row maximum.  Sampled:
 * q = softmax(row); the first slot whose cumulative mass exceeds u_walk (if
 * rounding leaves none, the last slot with q > 0).  q_sel records q (greedy:
 * one-hot).  A row with a NaN, or with every score -inf, ends the walk: that
 * position and the rest get token -1, slot -1 and NaN q.
 * margin[b,t]: greedy = best minus second-best score (inf if the rest are
 * -inf); sampled = smallest |cumulative mass - u| over the row.
 * R repetitions: u_walk is [R, B, K] and the outputs are [R, B, K(,16)].
 */
static void walk_one(int K, const int32_t *cand, const double *scores, double T, const float *u_walk,
                     int32_t *path_tok, int32_t *path_slot, double *q_sel, double *margin) {
    int prev = 0, dead = 0;
    for (int t = 0; t < K; t++) {
        double *q = q_sel ? q_sel + (int64_t)t * NC : NULL;
        const double *row = scores + ((int64_t)t * NC + prev) * NC;
        int bad = dead;
        double mx = -INFINITY;
        for (int j = 0; j < NC && !bad; j++) {
            if (isnan(row[j])) bad = 1;
            if (row[j] > mx) mx = row[j];
        }
        if (!bad && isinf(mx) && mx < 0) bad = 1;
        if (bad) {
            dead = 1;
            path_tok[t] = -1;
            path_slot[t] = -1;
            if (q)
                for (int j = 0; j < NC; j++) q[j] = NAN;
            if (margin) margin[t] = INFINITY;
            continue;
        }
        int js = -1;
        if (T == 0.0) {
            /* first maximal slot: strict comparison, scanning upwards */
            js = 0;
            for (int j = 1; j < NC; j++)
                if (row[j] > row[js]) js = j;
            double second = -INFINITY;
            for (int j = 0; j < NC; j++)
                if (j != js && row[j] > second) second = row[j];
            if (q)
                for (int j = 0; j < NC; j++) q[j] = (j == js) ? 1.0 : 0.0;
            if (margin) margin[t] = row[js] - second;
        } else {
            double e[NC], tot = 0.0;
            for (int j = 0; j < NC; j++) {
                e[j] = exp(row[j] - mx);
                tot += e[j];
            }
            double u = u_walk[t], cum = 0.0, mg = INFINITY;
            for (int j = 0; j < NC; j++) {
                cum += e[j];
                double d = fabs(cum / tot - u);
                if (d < mg) mg = d;
                if (js < 0 && cum > u * tot) js = j;
            }
            if (js < 0)
                for (int j = NC - 1; j >= 0; j--)
                    if (e[j] > 0.0) {
                        js = j;
                        break;
                    }
            if (q)
                for (int j = 0; j < NC; j++) q[j] = e[j] / tot;
            if (margin) margin[t] = mg;
        }
        path_slot[t] = js;
        path_tok[t] = cand[t * NC + js];
        prev = js;
    }
}

void dflash2_ref_walk(int64_t R, int64_t B, int K, const int32_t *cand_idx, const double *scores,
                      const float *temperature, const float *u_walk, int32_t *path_tok,
                      int32_t *path_slot, double *q_sel, double *margin) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t rep = 0; rep < R; rep++) {
        for (int64_t b = 0; b < B; b++) {
            int64_t o = (rep * B + b) * K;
            walk_one(K, cand_idx + b * K * NC, scores + b * K * NC * NC,
                     temperature ? temperature[b] : 0.0, u_walk ? u_walk + o : NULL, path_tok + o,
                     path_slot + o, q_sel ? q_sel + o * NC : NULL, margin ? margin + o : NULL);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* (5) target distribution of one verify row.                                */
/* ------------------------------------------------------------------------ */
/*
 * FreeToken PR 857 "Details"/Sampled verify and "Speed".  Greedy (T == 0):
 * all mass on the first maximal token.  Sampled: the filter above applied to
 * softmax(y/T).  Writes the support in rank order to ids/probs (cap entries
 * at most; the support is truncated to cap, which callers size to V or to
 * top_k) and returns its size, or -1 for an unusable row, or -2 for invalid
 * parameters.  *margin as in ref_filter.
 */
int64_t dflash2_ref_target_dist(const void *y, int dtype, int64_t V, float T, int32_t top_k,
                                 float top_p, int32_t *ids, double *probs, int64_t cap,
                                 double *margin) {
    double mg = INFINITY;
    if (params_bad(T, top_k, top_p)) return -2;
    if (row_is_bad(y, dtype, V)) return -1;
    if (T == 0.0f) {
        int64_t best = 0;
        double bv = ref_load(y, dtype, 0);
        for (int64_t v = 1; v < V; v++) {
            double z = ref_load(y, dtype, v);
            if (z > bv) {
                bv = z;
                best = v;
            }
        }
        ids[0] = (int32_t)best;
        probs[0] = 1.0;
        if (margin) *margin = mg;
        return 1;
    }
    entry *ord = sorted_row(y, dtype, V);
    double *prob = (double *)malloc((size_t)V * sizeof(double));
    double L;
    int64_t kept = ref_filter(ord, V, T, top_k, top_p, prob, &L, &mg);
    if (kept > cap) kept = cap;
    for (int64_t i = 0; i < kept; i++) {
        ids[i] = ord[i].id;
        probs[i] = prob[i];
    }
    free(prob);
    free(ord);
    if (margin) *margin = mg;
    return kept;
}

/* ------------------------------------------------------------------------ */
/* (6) speculative-sampling accept / residual resample of one request.       */
/* ------------------------------------------------------------------------ */
/*
 * FreeToken PR 857 "Details"/Sampled verify: accept with min(1, p/q); on a
 * reject resample from max(0, p - q); all-greedy requests keep the prefix
 * match.  DFlash 2 proposer issue "Proposal" phase 3 (greedy stays
 * longest-prefix; rejection sampling restores the exact target
 * distribution).
 *
 * dists: for t = 0..K, the target distribution of row t as (ids, probs, n);
 * rank order.  Accept position t iff u_acc[t] * q_d < p_d (u < p/q without a
 * division).  On a reject the residual r(v) = max(0, p(v) - q(v)), q(v) the
 * walk's probability of v among the candidates of position t, is drawn by
 * inverse CDF over v in ascending token id with u_res[t] (reading: the pages
 * give no order); if its total is <= 1e-12 the draw is from p.  After K
 * accepts the bonus token is drawn from row K with u_res[K].  Greedy requests
 * accept iff the drafted token is the target's argmax and emit the argmax.
 * margin: smallest |u*q - p| over the accept tests and smallest relative
 * |cum - u*Z| / Z over the inverse-CDF draws made.
 */
typedef struct {
    const int32_t *ids;
    const double *p;
    int64_t n;
} dist_t;

static double dist_prob(const dist_t *d, int32_t v) {
    for (int64_t i = 0; i < d->n; i++)
        if (d->ids[i] == v) return d->p[i];
    return 0.0;
}

/* inverse CDF over the support sorted by ascending id; weights w (>= 0). */
static int32_t draw_ascending(const int32_t *ids, const double *w, int64_t n, double u,
                              double *margin) {
    entry *e = (entry *)malloc((size_t)n * sizeof(entry));
    for (int64_t i = 0; i < n; i++) {
        e[i].id = ids[i];
        e[i].v = w[i];
    }
    qsort(e, (size_t)n, sizeof(entry), id_cmp);
    double Z = 0.0;
    for (int64_t i = 0; i < n; i++) Z += e[i].v;
    double cum = 0.0;
    int32_t pick = -1;
    for (int64_t i = 0; i < n; i++) {
        if (e[i].v <= 0.0) continue;
        cum += e[i].v;
        double d = fabs(cum - u * Z) / Z;
        if (d < *margin) *margin = d;
        if (pick < 0 && cum > u * Z) pick = e[i].id;
    }
    if (pick < 0)
        for (int64_t i = n - 1; i >= 0; i--)
            if (e[i].v > 0.0) {
                pick = e[i].id;
                break;
            }
    free(e);
    return pick;
}

static void accept_one(int K, const dist_t *dists, int greedy, const int32_t *path_tok,
                       const int32_t *cand, const double *q_sel, const int32_t *path_slot,
                       const float *u_acc, const float *u_res, int32_t *accept_len,
                       int32_t *out_tok, double *margin) {
    int n = 0;
    double mg = INFINITY;
    for (int t = 0; t <= K; t++) out_tok[t] = -1;
    for (int t = 0; t < K; t++) {
        const dist_t *d = &dists[t];
        int32_t tok = path_tok[t];
        if (greedy) {
            if (tok == d->ids[0]) {
                out_tok[n++] = tok;
                continue;
            }
            out_tok[n] = d->ids[0];
            *accept_len = n;
            if (margin) *margin = mg;
            return;
        }
        const double *q = q_sel + (int64_t)t * NC;
        double qd = q[path_slot[t]];
        double pd = dist_prob(d, tok);
        double lhs = (double)u_acc[t] * qd;
        if (fabs(lhs - pd) < mg) mg = fabs(lhs - pd);
        if (lhs < pd) {
            out_tok[n++] = tok;
            continue;
        }
        /* reject: residual max(0, p - q) over the support of p */
        double *r = (double *)malloc((size_t)d->n * sizeof(double));
        double Z = 0.0;
        for (int64_t i = 0; i < d->n; i++) {
            double qv = 0.0;
            for (int j = 0; j < NC; j++)
                if (cand[t * NC + j] == d->ids[i]) qv = q[j];
            r[i] = d->p[i] - qv > 0.0 ? d->p[i] - qv : 0.0;
            Z += r[i];
        }
        int32_t pick;
        if (Z <= 1e-12)
            pick = draw_ascending(d->ids, d->p, d->n, u_res[t], &mg);
        else
            pick = draw_ascending(d->ids, r, d->n, u_res[t], &mg);
        free(r);
        out_tok[n] = pick;
        *accept_len = n;
        if (margin) *margin = mg;
        return;
    }
    /* all K accepted: bonus token from row K */
    const dist_t *d = &dists[K];
    out_tok[K] = greedy ? d->ids[0] : draw_ascending(d->ids, d->p, d->n, u_res[K], &mg);
    *accept_len = K;
    if (margin) *margin = mg;
}

/* Request-level input checks shared by verify and the sparse accept below.
 * Sampled requests: q rows must be finite and non-negative (else NAN), sum to
 * 1 within 1e-3 unless trusted (else BAD_Q), and the drafted token must be
 * the candidate at its slot (else BAD_Q).  FreeToken PR 857 "Tests added or
 * changed" (trusted, NaN and wrong-total rows). */
static int check_q(int K, const int32_t *path_tok, const int32_t *cand, const double *q_sel,
                   const int32_t *path_slot, int trusted) {
    for (int t = 0; t < K; t++) {
        const double *q = q_sel + (int64_t)t * NC;
        double s = 0.0;
        for (int j = 0; j < NC; j++) {
            if (!isfinite(q[j]) || q[j] < 0.0) return REF_ST_NAN;
            s += q[j];
        }
        if (!trusted && fabs(s - 1.0) > 1e-3) return REF_ST_BAD_Q;
        int js = path_slot[t];
        if (js < 0 || js >= NC || cand[t * NC + js] != path_tok[t]) return REF_ST_BAD_Q;
    }
    return REF_ST_OK;
}

/*
 * Full verify: target distributions for the K+1 rows of each request, then
 * the accept walk.  tlogits is [B, K+1, V] with row stride ld.  A request with
 * an unusable target row gets status NAN, invalid parameters BAD_PARAMS, bad
 * q as in check_q; such a request commits nothing (accept_len 0, all -1).
 * margin[b]: the smallest margin of the decisions the request actually took:
 * the top_p cut of the target rows it used (rows 0..n, n = accept_len), its
 * accept tests and its draws (as in accept_one); inf for a request with a
 * nonzero status (its outcome is the status alone).
 */
void dflash2_ref_verify(const void *tlogits, int dtype, int64_t B, int K, int64_t V, int64_t ld,
                        const int32_t *path_tok, const int32_t *cand_idx, const double *q_sel,
                        const int32_t *path_slot, const float *temperature, const int32_t *top_k,
                        const float *top_p, const float *u_acc, const float *u_res, int trusted,
                        int32_t *accept_len, int32_t *out_tok, int32_t *status, double *margin) {
    size_t es = dtype == REF_BF16 ? 2 : 4;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t b = 0; b < B; b++) {
        double T = temperature ? temperature[b] : 0.0;
        int32_t tk = top_k ? top_k[b] : 0;
        double tp = top_p ? top_p[b] : 1.0;
        int greedy = T == 0.0;
        int st = REF_ST_OK;
        double mg = INFINITY;
        int32_t *ids = (int32_t *)malloc((size_t)(K + 1) * V * sizeof(int32_t));
        double *pr = (double *)malloc((size_t)(K + 1) * V * sizeof(double));
        dist_t *dists = (dist_t *)malloc((size_t)(K + 1) * sizeof(dist_t));
        double *row_mg = (double *)malloc((size_t)(K + 1) * sizeof(double));
        if (params_bad(T, tk, tp)) st = REF_ST_BAD_PARAMS;
        for (int t = 0; t <= K && st == REF_ST_OK; t++) {
            const void *row = (const char *)tlogits + (size_t)((b * (K + 1) + t) * ld) * es;
            double m1 = INFINITY;
            int64_t n = dflash2_ref_target_dist(row, dtype, V, (float)T, tk, (float)tp,
                                                ids + (int64_t)t * V, pr + (int64_t)t * V, V, &m1);
            if (n < 0) st = REF_ST_NAN;
            row_mg[t] = m1;
            dists[t].ids = ids + (int64_t)t * V;
            dists[t].p = pr + (int64_t)t * V;
            dists[t].n = n;
        }
        const int32_t *pt = path_tok + b * K;
        const int32_t *cd = cand_idx + b * K * NC;
        const double *qs = q_sel + b * K * NC;
        const int32_t *ps = path_slot + b * K;
        if (st == REF_ST_OK && !greedy) st = check_q(K, pt, cd, qs, ps, trusted);
        if (st != REF_ST_OK) {
            accept_len[b] = 0;
            for (int t = 0; t <= K; t++) out_tok[b * (K + 1) + t] = -1;
        } else {
            double m2 = INFINITY;
            accept_one(K, dists, greedy, pt, cd, qs, ps, u_acc + b * K, u_res + b * (K + 1),
                       &accept_len[b], out_tok + b * (K + 1), &m2);
            mg = m2;
            for (int t = 0; t <= accept_len[b]; t++)
                if (row_mg[t] < mg) mg = row_mg[t];
        }
        status[b] = st;
        if (margin) margin[b] = mg;
        free(row_mg);
        free(ids);
        free(pr);
        free(dists);
    }
}

/*
 * The accept walk alone over precomputed target distributions, for R
 * repetitions of the uniforms (Monte Carlo).  dist_ids/dist_p are
 * [B, K+1, cap] with dist_n [B, K+1]; u_acc [R, B, K], u_res [R, B, K+1];
 * outputs [R, B] and [R, B, K+1].  FreeToken PR 857 "Accuracy" (Monte Carlo
 * over 6M rows of the sampled verify).
 */
void dflash2_ref_accept_sparse(int64_t R, int64_t B, int K, const int32_t *dist_ids,
                               const double *dist_p, const int64_t *dist_n, int64_t cap,
                               const float *temperature, const int32_t *path_tok,
                               const int32_t *cand_idx, const double *q_sel,
                               const int32_t *path_slot, const float *u_acc, const float *u_res,
                               int trusted, int32_t *accept_len, int32_t *out_tok,
                               int32_t *status) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t rep = 0; rep < R; rep++) {
        for (int64_t b = 0; b < B; b++) {
            dist_t dists[64];
            int greedy = temperature ? temperature[b] == 0.0f : 1;
            for (int t = 0; t <= K; t++) {
                dists[t].ids = dist_ids + (b * (K + 1) + t) * cap;
                dists[t].p = dist_p + (b * (K + 1) + t) * cap;
                dists[t].n = dist_n[b * (K + 1) + t];
            }
            const int32_t *pt = path_tok + b * K;
            const int32_t *cd = cand_idx + b * K * NC;
            const double *qs = q_sel + b * K * NC;
            const int32_t *ps = path_slot + b * K;
            int64_t o = rep * B + b;
            int st = greedy ? REF_ST_OK : check_q(K, pt, cd, qs, ps, trusted);
            status[o] = st;
            if (st != REF_ST_OK) {
                accept_len[o] = 0;
                for (int t = 0; t <= K; t++) out_tok[o * (K + 1) + t] = -1;
                continue;
            }
            accept_one(K, dists, greedy, pt, cd, qs, ps, u_acc + o * K, u_res + o * (K + 1),
                       &accept_len[o], out_tok + o * (K + 1), NULL);
        }
    }
}

/*
 * Monte Carlo of the whole selection + verify decision: for each of R
 * repetitions, a fresh sampled walk over the fixed scores (u_walk [R, B, K])
 * and then the accept walk over the fixed target distributions (u_acc
 * [R, B, K], u_res [R, B, K+1]).  Outputs accept_len [R, B], out_tok
 * [R, B, K+1].  FreeToken PR 857 "Accuracy" (committed-token marginals within
 * 5e-3 of the target distribution over 6M rows).
 */
void dflash2_ref_walk_accept_mc(int64_t R, int64_t B, int K, const int32_t *cand_idx,
                                const double *scores, const float *temperature,
                                const int32_t *dist_ids, const double *dist_p,
                                const int64_t *dist_n, int64_t cap, const float *u_walk,
                                const float *u_acc, const float *u_res, int32_t *accept_len,
                                int32_t *out_tok) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t rep = 0; rep < R; rep++) {
        for (int64_t b = 0; b < B; b++) {
            int32_t pt[64], ps[64];
            double q[64 * NC];
            dist_t dists[64];
            double T = temperature ? temperature[b] : 0.0;
            int64_t o = rep * B + b;
            const int32_t *cd = cand_idx + b * K * NC;
            walk_one(K, cd, scores + b * K * NC * NC, T, u_walk + o * K, pt, ps, q, NULL);
            for (int t = 0; t <= K; t++) {
                dists[t].ids = dist_ids + (b * (K + 1) + t) * cap;
                dists[t].p = dist_p + (b * (K + 1) + t) * cap;
                dists[t].n = dist_n[b * (K + 1) + t];
            }
            accept_one(K, dists, T == 0.0, pt, cd, q, ps, u_acc + o * K, u_res + o * (K + 1),
                       &accept_len[o], out_tok + o * (K + 1), NULL);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* (7) two-tap dynamic depthwise convolution.                                */
/* ------------------------------------------------------------------------ */
/* Round a double to the nearest bf16 value, ties to even (8 significant bits,
 * f32 exponent range, bf16 subnormals below 2^-126). */
static double round_bf16(double v) {
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    double a = fabs(v);
    double q; /* spacing of bf16 values around a */
    if (a < ldexp(1.0, -126)) {
        q = ldexp(1.0, -133);
    } else {
        int e;
        frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
        q = ldexp(1.0, e - 8);
    }
    double r = nearbyint(a / q) * q; /* a / q is exact: q is a power of two */
    if (r > 3.38953138925153547590470800371487866880e38) r = INFINITY; /* above max bf16 */
    return v < 0 ? -r : r;
}

static double round_f32(double v) { return (double)(float)v; }

/* Exact a + b rounded once by `rnd`.  a and b are exact products (two 8- or
 * 24-bit significands fit a double), and two-sum gives a + b = s + e exactly
 * with |e| at most half an ulp of s.  Rounding s instead of s + e can only go
 * wrong when s is exactly a midpoint of the target format (its two double
 * neighbours round apart); then the sign of e picks the side. */
static double round_sum(double a, double b, double (*rnd)(double)) {
    double s = a + b;
    double bb = s - a;
    double e = (a - (s - bb)) + (b - bb);
    if (e != 0.0) {
        double below = rnd(nextafter(s, -INFINITY)), above = rnd(nextafter(s, INFINITY));
        if (below != above) return e > 0 ? above : below;
    }
    return rnd(s);
}

/*
 * DFlash 2 proposer issue, "What upstream shipped" item 2:
 * Conv(x)_t = k_{t,0} * x_t + k_{t,1} * x_{t-1}, the first position tapping
 * the last verified token's hidden (x_prev).  FreeToken PR 857 "Details"
 * (conv_group_size divides the hidden size): with group size G the taps are
 * shared by G adjacent channels, k shaped [B, T, H/G].  The output is the
 * exact value rounded once to the I/O dtype (nearest, ties to even).
 */
void dflash2_ref_conv2tap(const void *x, const void *k0, const void *k1, const void *x_prev,
                          int dtype, int64_t B, int T, int64_t H, int G, void *y) {
    int64_t Hk = H / G;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; b++) {
        for (int t = 0; t < T; t++) {
            for (int64_t c = 0; c < H; c++) {
                int64_t o = (b * T + t) * H + c;
                int64_t ko = (b * T + t) * Hk + c / G;
                double xc = ref_load(x, dtype, o);
                double xp = t == 0 ? ref_load(x_prev, dtype, b * H + c)
                                   : ref_load(x, dtype, o - H);
                double a = ref_load(k0, dtype, ko) * xc;
                double bb = ref_load(k1, dtype, ko) * xp;
                if (dtype == REF_BF16) {
                    double r = round_sum(a, bb, round_bf16);
                    float f = (float)r;
                    uint32_t u;
                    memcpy(&u, &f, 4);
                    ((uint16_t *)y)[o] = (uint16_t)(u >> 16);
                } else {
                    ((float *)y)[o] = (float)round_sum(a, bb, round_f32);
                }
            }
        }
    }
}

/*
 * Grouped dynamic taps.  The pages give the conv's form, "dynamic", and the
 * group size (conv_group_size divides the hidden size), not how the taps are
 * made; the reading here is dynamic convolution as published (Wu et al.,
 * "Pay Less Attention with Lightweight and Dynamic Convolutions", 2019):
 * position t's taps are a linear map of its own input, normalised by a
 * softmax over the kernel's width and shared by the G channels of a group.
 * With two taps, softmax(a0, a1) = (s, 1 - s) with s = sigmoid(a0 - a1), so
 * the map enters through its difference Wd = W0 - W1, [H/G, H]:
 *   k_{t,0}[g] = sigmoid(Wd[g] . x_t),  k_{t,1}[g] = 1 - k_{t,0}[g],
 *   y_t[c] = k_{t,0}[c / G] x_t[c] + k_{t,1}[c / G] x_{t-1}[c]
 * (x_prev at t = 0).  taps receives k_{t,0} in fp64, [B, T, H/G]; y is the
 * fp64 value rounded once to the I/O dtype (nearest, ties to even).
 */
void dflash2_ref_dynconv2tap(const void *x, const void *x_prev, const void *Wd, int dtype, int64_t B, int T,
                             int64_t H, int G, double *taps, void *y) {
    int64_t Hk = H / G;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; b++) {
        for (int t = 0; t < T; t++) {
            int64_t row = b * T + t;
            for (int64_t g = 0; g < Hk; g++) {
                double a = 0.0;
                for (int64_t c = 0; c < H; c++) a += ref_load(Wd, dtype, g * H + c) * ref_load(x, dtype, row * H + c);
                taps[row * Hk + g] = 1.0 / (1.0 + exp(-a));
            }
            for (int64_t c = 0; c < H; c++) {
                int64_t o = row * H + c;
                double k0 = taps[row * Hk + c / G], k1 = 1.0 - k0;
                double xc = ref_load(x, dtype, o);
                double xp = t == 0 ? ref_load(x_prev, dtype, b * H + c) : ref_load(x, dtype, o - H);
                double v = k0 * xc + k1 * xp;
                if (dtype == REF_BF16) {
                    float f = (float)round_bf16(v);
                    uint32_t u;
                    memcpy(&u, &f, 4);
                    ((uint16_t *)y)[o] = (uint16_t)(u >> 16);
                } else {
                    ((float *)y)[o] = (float)v;
                }
            }
        }
    }
}

int dflash2_ref_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void dflash2_ref_set_num_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n);
#else
    (void)n;
#endif
}
