/*
 * dflash2.h -- C ABI of the DFlash 2 draft-selection + verify path on one GPU.
 *
 * The DFlash 2 proposer keeps the 16 best candidates of every drafted
 * position, scores adjacent candidate pairs with a low-rank bilinear term
 * gated by the drafter's hidden state, walks those scores once to pick the
 * proposed path, and the verify accepts drafted tokens with probability
 * min(1, p/q) and resamples a rejected one from max(0, p - q).  Sources:
 *   [P] "qwen3/dflash: DFlash 2 proposer -- top-16 path selector + two-tap
 *       dynamic convolution" (pegainfer issue 930): "What upstream shipped"
 *       items 1-2, "Proposal" phases 1-3.
 *   [F] FreeToken PR 857 (DFlash 2 next to MTP): "Details" (Runtime, Sampled
 *       verify, Refused at startup), "Tests added or changed", "Known gaps".
 *
 * Conventions shared by every entry point
 *   - Tensor arguments are DEVICE pointers owned by the caller, row-major and
 *     16-byte aligned.  Nothing here allocates, frees or synchronises: each
 *     call enqueues its kernels on `stream` and returns.
 *   - A call returns DFLASH2_ERR_INVALID_ARG before launching anything when an
 *     argument is out of range (see each call); DFLASH2_ERR_CUDA when a launch
 *     fails (the CUDA error is left for cudaGetLastError).
 *   - Per-request data problems never abort a batch: they are reported per
 *     request in `status` (DFLASH2_ST_*) or as -1 / NaN outputs.
 *   - Workspaces (`ws`) are caller-provided device buffers of at least the
 *     size returned by the matching *_workspace_bytes function.  They must be
 *     zero-filled once before first use; every call that runs to the end
 *     leaves them zeroed again.  After a call that returned DFLASH2_ERR_CUDA,
 *     or after dflash2_device_error reported a nonzero code (a kernel gave up
 *     on a bounded wait), zero-fill the workspaces of the calls involved
 *     again before reusing them.  Two calls that share a workspace must not
 *     run concurrently.
 *   - The first call on a device performs one-time set-up (device attributes,
 *     kernel attributes); make it before any stream capture.  Later calls are
 *     capturable into CUDA graphs.
 *   - Ties in logits are broken by the lower token id everywhere.
 */
#ifndef DFLASH2_H
#define DFLASH2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *dflash2_stream;

typedef enum {
    DFLASH2_OK = 0,
    DFLASH2_ERR_INVALID_ARG = 1,
    DFLASH2_ERR_UNSUPPORTED = 2,
    DFLASH2_ERR_CUDA = 3,
    DFLASH2_ERR_WORKSPACE = 4
} dflash2_status;

typedef enum { DFLASH2_F32 = 0, DFLASH2_BF16 = 1 } dflash2_dtype;

/* Per-request verify status. */
enum {
    DFLASH2_ST_OK = 0,
    DFLASH2_ST_NAN = 1,         /* NaN or +Inf (or no value above -Inf) in a target row; NaN, Inf or
                                   a negative value in a q row */
    DFLASH2_ST_BAD_Q = 2,       /* a q row does not sum to 1 within 1e-3, or a drafted token is not
                                   the candidate at its slot */
    DFLASH2_ST_BAD_PARAMS = 3,  /* temperature < 0 or not finite, top_k < 0, top_p outside (0, 1] */
    DFLASH2_ST_UNSUPPORTED = 4  /* kept for the ABI: no parameters produce it any more */
};

#define DFLASH2_NC 16        /* candidates per draft position ([P] item 1) */
#define DFLASH2_MAX_K 15     /* drafted positions: [F] Details refuses k outside 1 .. block_size - 1; the pages
                                set no bound on block_size, and the cap of 15 (block_size <= 16) is this
                                library's own limit, not a number the pages print */
#define DFLASH2_MAX_TOPK 64  /* top_k up to this is taken from the row's best-key list in one pass;
                                larger top_k, or top_p with top_k off, need further passes */

/*
 * Sampling parameters of one request, applied to draft and target alike in
 * the order temperature -> top_k -> renormalise -> top_p -> renormalise
 * ([F] "Speed": temperature 1.0, top_p 0.95, top_k 20 on both sides).
 * temperature == 0 is greedy.  top_k == 0 (or >= V) and top_p == 1 switch the
 * filters off.  Every combination is supported.  With top_k <= 64 the row's
 * best-key list settles the filter in one pass; with top_k above 64, or top_p
 * with top_k off, the kept prefix may reach further and the cut is found by
 * passes over the row (dflash2_topk16, dflash2_verify).  The fused LM head
 * and the vocabulary-sharded merge take only rows settled by 16 or 64 best
 * tokens and give the others -1 / NaN.
 */
typedef struct {
    float temperature;
    int32_t top_k;
    float top_p;
} dflash2_sampling;

/*
 * dflash2_topk16 -- [P] item 1 "keep top-16 candidates per position"; [F]
 * Runtime "the target LM head gives 16 candidates per slot".
 *
 * logits   [rows, ld] of dt (row stride ld elements, ld >= V, ld * elem
 *          size a multiple of 16 bytes); the first V entries of a row count.
 * params   device [ceil(rows / rows_per_param)] or NULL (all greedy); row r
 *          uses params[r / rows_per_param].
 * cand_idx [rows, 16] int32: the 16 best tokens, best first.
 * cand_U   [rows, 16] f32: log-probability of each candidate under the
 *          drafter's distribution: greedy rows log softmax(z), sampled rows
 *          log of the filtered softmax(z / T), -inf for a candidate the
 *          filter drops.
 * lse      [rows] f32: the log normaliser on the z / T' scale (T' = 1 for
 *          greedy rows), so that kept candidates have U = z / T' - lse.
 * A row holding a NaN or +Inf, or nothing above -Inf, or with invalid
 * parameters, gets cand_idx -1, U NaN and lse NaN.  Every filter is
 * supported: a row whose kept prefix reaches past its 64 best tokens (top_k
 * above 64, or top_p with top_k off) is finished with further passes over
 * the row (a radix select of the cut by count and by mass), in the same
 * kernel: the CTA that completes such a row finishes it once it has
 * streamed its share of the rows.
 * ws: dflash2_topk16_workspace_bytes(rows) bytes (the kernel splits long rows
 *   over several CTAs and combines the parts there, and marks there the rows
 *   a CTA finishes after its stream).
 * Errors: INVALID_ARG if a pointer is NULL or misaligned, rows < 0, V < 16,
 * V >= 2^31, ld < V, ld * elem size not a multiple of 16, rows_per_param < 1;
 * WORKSPACE if ws_bytes is too small.
 */
size_t dflash2_topk16_workspace_bytes(int64_t rows);
dflash2_status dflash2_topk16(const void *logits, dflash2_dtype dt, int64_t rows, int64_t V,
                              int64_t ld, const dflash2_sampling *params, int64_t rows_per_param,
                              int32_t *cand_idx, float *cand_U, float *lse, void *ws,
                              size_t ws_bytes, dflash2_stream stream);

/*
 * dflash2_topk16_noalloc -- no counterpart on the pages: an addition of this
 * library.  The same computation, arguments and argument errors as
 * dflash2_topk16, without the workspace, for callers that cannot give this
 * library device memory: a plugin, or an engine whose memory pool owns all
 * device memory and hands no scratch to the code it calls, or code that may
 * not call an allocator at the point where the drafter's rows are reduced.
 * The scratch (one ticket and one mark per row, and the partial records of
 * rows that the kernel splits over several CTAs) is a fixed array in the
 * library's own device memory, sized for
 * DFLASH2_TOPK16_NOALLOC_MAX_ROWS rows (about 1.2 MB),
 * held by every GPU that loads the library until the process exits.
 *   - rows > DFLASH2_TOPK16_NOALLOC_MAX_ROWS returns DFLASH2_ERR_WORKSPACE and
 *     launches nothing.
 *   - Nothing is allocated.  The tickets must start at zero: each call clears
 *     those of its rows (cudaMemsetAsync on `stream`) before the kernel.  The
 *     partial records are written before they are read.
 *   - The first call on a device looks up the array's device address (once,
 *     with that device current); make that first call before any stream
 *     capture.
 *   - All calls share the one array: calls that overlap on the GPU (on
 *     different streams, or from different threads) race on it and their
 *     outputs are undefined.  Issue them on one stream.
 */
#define DFLASH2_TOPK16_NOALLOC_MAX_ROWS 16384
dflash2_status dflash2_topk16_noalloc(const void *logits, dflash2_dtype dt, int64_t rows, int64_t V,
                                      int64_t ld, const dflash2_sampling *params, int64_t rows_per_param,
                                      int32_t *cand_idx, float *cand_U, float *lse, dflash2_stream stream);

/*
 * Vocabulary-sharded top-16 -- no counterpart on the pages, which run the
 * drafter with --tp 1 ([F] Known gaps): an addition of this library for an
 * LM head split over GPUs by vocabulary.  Each GPU reduces its slice of the
 * vocabulary to a partial (dflash2_topk16_shard); the partials of all slices
 * are exchanged once (an all-gather of DFLASH2_SHARD_LIST * 8 + 8 bytes per
 * row and slice, done by the caller); dflash2_topk16_merge then gives the
 * outputs dflash2_topk16 gives for the whole row, with the same sampling
 * parameters (top_k and top_p refer to the whole vocabulary V_total).
 *
 * dflash2_topk16_shard: logits [rows, ld] of dt hold tokens id_offset ..
 *   id_offset + V_shard - 1 of each row (V_shard >= 16).  Outputs:
 *   part_idx [rows, DFLASH2_SHARD_LIST] int32: the slice's best tokens in
 *     rank order as global ids, as many as the row needs (16; max(16, top_k)
 *     for a top_k-filtered row), -1 after;
 *   part_z [rows, DFLASH2_SHARD_LIST] f32: their logits, -inf after;
 *   part_m [rows] f32: the slice's largest logit;
 *   part_s [rows] f32: the sum over the slice of exp((z - part_m) / T'), T'
 *     the temperature (1 for greedy rows); 0 for filtered rows.
 *   A row with a NaN or +Inf in the slice, invalid parameters, or a filter
 *   that needs the whole row (top_k above 64, or top_p with top_k off), gets
 *   -1 ids and NaN m and s.  A slice of masked tokens (all
 *   -inf) is not an error: m = -inf, s = 0.
 *   ws: dflash2_topk16_workspace_bytes(rows).  Errors: those of dflash2_topk16
 *   (with V_shard as V), and INVALID_ARG for id_offset < 0 or
 *   id_offset + V_shard > V_total.
 *
 * dflash2_topk16_merge: the partials of the S slices laid out [S, rows, ...]
 *   (slice s at s * rows * DFLASH2_SHARD_LIST and s * rows); params and
 *   rows_per_param as for dflash2_topk16.  Outputs cand_idx, cand_U, lse as
 *   dflash2_topk16's for the whole rows (lse and U equal up to fp32 rounding:
 *   the log normaliser is summed per slice).  A row with a NaN partial or no
 *   finite largest logit gets -1 / NaN.  Errors: INVALID_ARG for S outside
 *   1..DFLASH2_MAX_SHARDS, rows < 0, V_total < 16, NULL pointers.
 */
#define DFLASH2_SHARD_LIST 64
#define DFLASH2_MAX_SHARDS 1024
dflash2_status dflash2_topk16_shard(const void *logits, dflash2_dtype dt, int64_t rows, int64_t V_shard, int64_t ld,
                                    int64_t id_offset, int64_t V_total, const dflash2_sampling *params,
                                    int64_t rows_per_param, int32_t *part_idx, float *part_z, float *part_m,
                                    float *part_s, void *ws, size_t ws_bytes, dflash2_stream stream);
dflash2_status dflash2_topk16_merge(int32_t S, int64_t rows, const int32_t *part_idx, const float *part_z,
                                    const float *part_m, const float *part_s, int64_t V_total,
                                    const dflash2_sampling *params, int64_t rows_per_param, int32_t *cand_idx,
                                    float *cand_U, float *lse, dflash2_stream stream);

/*
 * dflash2_lmhead_topk16 -- the drafter's LM head fused with dflash2_topk16:
 * [P] "What upstream shipped" item 1 (keep the top-16 candidates of each
 * drafted position) and [F] Runtime (16 candidates per slot from the LM
 * head), with the logits z = h . W^T never written to memory.  The GEMM runs
 * on the tensor cores (bf16 inputs, fp32 accumulation); the candidates, U
 * and lse are those of dflash2_topk16 on the fp32 logits.
 *
 * h [rows, hidden] bf16 and W [V, hidden] bf16, row-major (W is the LM head's
 * weight, one row per token).  hidden a multiple of 64.  params and
 * rows_per_param as for dflash2_topk16.  Rows that would need more than 16
 * candidates (a top_k filter above 16) or the whole row (top_p with top_k
 * off) get -1 / NaN.
 * ws: dflash2_lmhead_topk16_workspace_bytes(rows, V) bytes, for the current
 *   device (the per-row partials of each CTA's vocabulary range, combined by
 *   dflash2_topk16_merge on the same stream).
 * Errors: INVALID_ARG for NULL or misaligned pointers, rows < 0, hidden not a
 * positive multiple of 64, V < 16 or V >= 2^31, rows_per_param < 1;
 * WORKSPACE if ws_bytes is too small.
 */
size_t dflash2_lmhead_topk16_workspace_bytes(int64_t rows, int64_t V);
dflash2_status dflash2_lmhead_topk16(const void *h, const void *W, int64_t rows, int64_t hidden, int64_t V,
                                     const dflash2_sampling *params, int64_t rows_per_param, int32_t *cand_idx,
                                     float *cand_U, float *lse, void *ws, size_t ws_bytes, dflash2_stream stream);

/*
 * dflash2_ctx_gate -- [P] item 1 "context gate" of the bilinear selector,
 * taken as gate = sigmoid(W_g h) with no bias.
 *
 * h     [n, hidden] of dt;  Wg [D, hidden] of dt;  gate [n, D] f32.
 * bf16 runs on the tensor cores (fp32 accumulation); f32 on the CUDA cores.
 * The bf16 grid may start while the previous kernel in the stream still
 * runs, once that kernel allows it (programmatic dependent launch; of this
 * library's kernels, the row scans allow it at their start), so that it
 * overlaps dflash2_topk16's tail: h and Wg must not be written by the
 * kernel just before it.  It completes only after that kernel does.
 * Errors: INVALID_ARG if a pointer is NULL or misaligned, n < 0, D not in
 * {16, 32, ..., 512} (a power of two), hidden < 1, or (bf16) hidden not a
 * multiple of 64.
 */
dflash2_status dflash2_ctx_gate(const void *h, dflash2_dtype dt, int64_t n, int64_t hidden,
                                const void *Wg, int32_t D, float *gate, dflash2_stream stream);

/*
 * dflash2_pair_score_walk -- [P] item 1 (S_t(a,b) = U_t(b) + <A(a) * H(h_t),
 * B(b)>, one greedy or sampled walk over the precomputed scores) and
 * "Proposal" phase 1 (block_size x 16 preds x 16 cands x 256 dims, a
 * <= block_size-step argmax walk); [F] Runtime (sampled from q, argmax when
 * greedy).
 *
 * cand_idx [B, K, 16] int32, cand_U [B, K, 16] f32 (from dflash2_topk16).
 * last_tok [B] int32: the last verified token, the only predecessor at t = 0.
 * A, Bt    [V, D] of tdt: the two token-embedding tables.
 * gate     [B, K, D] f32 (from dflash2_ctx_gate).
 * params   [B] or NULL (all greedy); only temperature is read (0 = greedy).
 * u_walk   [B, K] f32 uniforms in [0, 1); may be NULL when params is NULL.
 * Outputs: path_tok [B, K] int32, path_slot [B, K] int32 (index into the
 *   candidates), q_sel [B, K, 16] f32 (the walk's distribution at each step;
 *   one-hot when greedy), scores [B, K, 16, 16] f32: scores[b,t,i,j] pairs
 *   predecessor i with candidate j; at t = 0 row 0 is the last verified
 *   token and rows 1..15 are -inf.
 * Greedy steps take the first slot with the largest score; sampled steps
 * take the first slot whose cumulative q exceeds u_walk.  A step whose row
 * holds a NaN, or only -inf, ends the walk: that step and the rest get
 * token -1, slot -1 and NaN q.  Ids outside [0, V) give NaN scores.
 * No workspace: one thread-block cluster of K CTAs per request keeps the
 *   request's state in its shared memory.
 * Errors: INVALID_ARG for NULL/misaligned pointers, B < 0, K outside 1..15,
 * D not a power of two in 16..1024, V < 16, u_walk NULL with params set;
 * UNSUPPORTED for B > 65535, or when a cluster of K CTAs with the shared
 * memory that D needs cannot be resident on this GPU (clusters above 8 CTAs
 * must fit in one GPC; the answer is cached per device, K and D).
 */
dflash2_status dflash2_pair_score_walk(int64_t B, int32_t K, const int32_t *cand_idx,
                                       const float *cand_U, const int32_t *last_tok,
                                       const void *A, const void *Bt, dflash2_dtype tdt, int64_t V,
                                       int32_t D, const float *gate,
                                       const dflash2_sampling *params, const float *u_walk,
                                       int32_t *path_tok, int32_t *path_slot, float *q_sel,
                                       float *scores, dflash2_stream stream);

/*
 * dflash2_verify -- [F] Sampled verify (accept with min(1, p/q); on a reject
 * resample from max(0, p - q); all-greedy batches keep the prefix match);
 * [P] "Proposal" phase 3; [F] "Tests added or changed" (trusted, NaN,
 * wrong-total and greedy rows).
 *
 * tlogits [B, K+1, ld] of dt: target logits of the K drafted positions and
 *   the bonus position, row (b, t) at (b * (K+1) + t) * ld.
 * path_tok, path_slot [B, K]; cand_idx, q_sel [B, K, 16] (from the walk).
 * params [B] or NULL (all greedy).  u_acc [B, K], u_res [B, K+1] f32
 *   uniforms in [0, 1); may be NULL when params is NULL.
 * flags: DFLASH2_VERIFY_TRUST_Q skips the q-total check.
 * Per request b: p_t is the target distribution of row t (greedy: all mass
 *   on the argmax).  Greedy requests accept while the drafted token is the
 *   argmax and then emit the argmax.  Sampled requests accept position t iff
 *   u_acc[t] * q < p at the drafted token; on a reject they draw from
 *   max(0, p - q) (normalised; from p when its total is <= 1e-12) by inverse
 *   CDF over ascending token ids with u_res[t]; after K accepts they draw the
 *   bonus token from p_K with u_res[K].  Every filter is supported: when
 *   p's support reaches past the row's 64 best tokens (no filter, top_p with
 *   top_k off, top_k above 64), the cut is found by further passes over the
 *   row and the residual and bonus draws walk the whole row in token-id order,
 *   in the same kernel, by the CTA that completes the row once it has
 *   streamed its share of the rows.
 * Outputs: accept_len [B] in 0..K; out_tok [B, K+1]: the accepted tokens,
 *   then the corrected or bonus token, then -1; status [B] (DFLASH2_ST_*).
 *   A request with status != 0 commits nothing (accept_len 0, all -1).
 * ws: dflash2_verify_workspace_bytes(B, K).
 * Errors: INVALID_ARG as for dflash2_topk16 plus K outside 1..15 and NULL
 * uniforms with params set.
 */
#define DFLASH2_VERIFY_TRUST_Q 1u
size_t dflash2_verify_workspace_bytes(int64_t B, int32_t K);
dflash2_status dflash2_verify(const void *tlogits, dflash2_dtype dt, int64_t B, int32_t K,
                              int64_t V, int64_t ld, const int32_t *path_tok,
                              const int32_t *cand_idx, const float *q_sel,
                              const int32_t *path_slot, const dflash2_sampling *params,
                              const float *u_acc, const float *u_res, uint32_t flags,
                              int32_t *accept_len, int32_t *out_tok, int32_t *status, void *ws,
                              size_t ws_bytes, dflash2_stream stream);

/*
 * dflash2_conv2tap -- [P] item 2: Conv(x)_t = k_{t,0} * x_t + k_{t,1} * x_{t-1},
 * the first position tapping the last verified token's hidden state; [F]
 * Refused at startup (conv_group_size divides the hidden size).
 *
 * x [B, T, H], k0 and k1 [B, T, H / group_size], x_prev [B, H], y [B, T, H],
 * all of dt.  With group_size G, channel c uses tap c / G.  bf16 outputs are
 * the exact value rounded once to bf16 (nearest, ties to even); f32 outputs
 * use one fused multiply-add.
 * Errors: INVALID_ARG for NULL/misaligned pointers, B < 0, T < 1, H < 1,
 * group_size < 1 or not dividing H.
 */
dflash2_status dflash2_conv2tap(const void *x, const void *k0, const void *k1, const void *x_prev,
                                dflash2_dtype dt, int64_t B, int32_t T, int64_t H,
                                int32_t group_size, void *y, dflash2_stream stream);

/*
 * dflash2_dynconv2tap -- [P] item 2 with the taps made from the input: the
 * pages name the conv "dynamic" and give its group size ([F] Refused at
 * startup: conv_group_size divides the hidden size), not how the taps are
 * made.  The reading is dynamic convolution as published (Wu et al., "Pay
 * Less Attention with Lightweight and Dynamic Convolutions", 2019): the
 * taps of position t are a linear map of x_t, normalised by a softmax over
 * the kernel's width and shared by the group_size channels of a group.  For
 * two taps that softmax is (s, 1 - s) with s = sigmoid(a0 - a1), so the map
 * enters through its difference Wd:
 *   taps[b, t, g] = k0 = sigmoid(Wd[g] . x[b, t]),  k1 = 1 - k0,
 *   y[b, t, c] = k0 x[b, t, c] + k1 x[b, t-1, c]   (x_prev at t = 0, g = c / group_size).
 *
 * x [B, T, H], x_prev [B, H], Wd [H / group_size, H], y [B, T, H], all of dt;
 * taps [B, T, H / group_size] f32 (an output).  bf16: the taps on the tensor
 * cores (fp32 accumulation) as dflash2_ctx_gate computes its gate; y is
 * fma(k0, x_t, k1 x_{t-1}) in fp32 rounded once to bf16 (within one bf16 ulp
 * of the exact value).  f32: CUDA cores, y by one fused multiply-add.
 * Not built: fusing the conv with the drafter sublayer's norm and residual
 * (the pages give no form for them).
 * Errors: INVALID_ARG for NULL/misaligned pointers (x, Wd, taps 16-byte
 * aligned), B < 0, T < 1, H < 1, group_size < 1 or not dividing H;
 * UNSUPPORTED for bf16 unless H is a multiple of 64 and H / group_size a
 * power of two in 16..512.
 */
dflash2_status dflash2_dynconv2tap(const void *x, const void *x_prev, const void *Wd, dflash2_dtype dt,
                                   int64_t B, int32_t T, int64_t H, int32_t group_size, float *taps, void *y,
                                   dflash2_stream stream);

/* Human-readable name of a status code (static string). */
const char *dflash2_status_string(dflash2_status s);

/*
 * Error word of the library's kernels on the current device: nonzero after a
 * kernel gave up on a bounded wait (it then wrote -1 / NaN outputs instead of
 * hanging; the word then holds DFLASH2_DEVERR_WAIT_TIMEOUT).  Synchronises
 * the device.  clear != 0 resets the word.
 */
#define DFLASH2_DEVERR_WAIT_TIMEOUT 1u
dflash2_status dflash2_device_error(uint32_t *code, int clear);

/*
 * dflash2_test_hold -- no counterpart on the pages: a test hook of this
 * library, for exercising the bounded waits without a GPU fault.  With `flag`
 * set (a 4-byte aligned device word), every streaming warp of every
 * dflash2_topk16 / dflash2_topk16_noalloc / dflash2_verify kernel launched
 * afterwards by this process first waits until *flag is nonzero, giving up
 * after max_cycles SM clock cycles (1 .. 2^32).  A warp that gives up issues
 * no copy, sets the device error word (DFLASH2_DEVERR_WAIT_TIMEOUT) and goes
 * through its rows as after any time-out: their outputs are -1 / NaN, and a
 * verify request that reads such a row gets status DFLASH2_ST_NAN.  flag NULL
 * switches the hook off.  Kernels already launched or captured keep the
 * setting they were launched with.
 * Errors: INVALID_ARG for a misaligned flag or max_cycles out of range.
 */
dflash2_status dflash2_test_hold(const uint32_t *flag, int64_t max_cycles);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H */
