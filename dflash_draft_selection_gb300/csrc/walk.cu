// walk.cu -- dflash2_pair_score_walk: the path selector.
//
// DFlash 2 proposer issue, "What upstream shipped" item 1: score every
// adjacent candidate pair S_t(a,b) = U_t(b) + <A(a) * H(h_t), B(b)> (256-dim
// token embeddings and a context gate: a low-rank bilinear attention) and
// pick the proposed path with a single greedy or sampled walk over the
// precomputed scores; "Proposal" phase 1 (block_size x 16 preds x 16 cands x
// 256 dims, a <= block_size-step argmax walk).  FreeToken PR 857,
// "Details"/Runtime (the path is sampled from q, or argmax when greedy).
//
// One CTA per (request, position) gathers the 16 candidate rows of B and the
// predecessor rows of A (16 candidates of the previous position, or the last
// verified token at t = 0), scales A by the gate and computes the 16 x 16
// score tile with fp32 FMAs from shared memory.  The CTA that finishes a
// request's last tile (atomic ticket) walks the K tiles.
#include "host.hpp"
#include "common.cuh"

namespace dfl {

constexpr int WALK_THREADS = 256;

struct WalkArgs {
    int64_t B;
    int K;
    int64_t V;
    int D;
    const int32_t *cand_idx;
    const float *cand_U;
    const int32_t *last_tok;
    const void *A;
    const void *Bt;
    const float *gate;
    const dflash2_sampling *params;
    const float *u_walk;
    int32_t *path_tok;
    int32_t *path_slot;
    float *q_sel;
    float *scores;
    int32_t *tickets;
};

template <bool BF16>
__device__ __forceinline__ void load_row_chunk(const void *table, int64_t row, int D, int k, float (&v)[4]) {
    if (BF16) {
        const uint2 w = *reinterpret_cast<const uint2 *>(static_cast<const unsigned short *>(table) +
                                                         row * D + k);
        v[0] = bf16lo(w.x);
        v[1] = bf16hi(w.x);
        v[2] = bf16lo(w.y);
        v[3] = bf16hi(w.y);
    } else {
        const float4 f = *reinterpret_cast<const float4 *>(static_cast<const float *>(table) + row * D + k);
        v[0] = f.x;
        v[1] = f.y;
        v[2] = f.z;
        v[3] = f.w;
    }
}

// The walk of request b by one warp over its K score tiles in shared memory.
__device__ void walk_request(const WalkArgs &a, int64_t b, const float *sS, const int32_t *sC, int lane) {
    const int K = a.K;
    const float T = a.params ? a.params[b].temperature : 0.0f;
    const bool greedy = !(T > 0.0f);
    int prev = 0;
    bool dead = false;
    for (int t = 0; t < K; ++t) {
        const float v = lane < NC ? sS[(t * NC + prev) * NC + lane] : NEG_INF;
        const int64_t o = b * K + t;
        const bool isn = lane < NC && v != v;
        float mx = v;
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, d));
        dead = dead || __any_sync(FULL, isn) || mx == NEG_INF;
        if (dead) {
            if (lane < NC) a.q_sel[o * NC + lane] = NAN;
            if (lane == 0) {
                a.path_tok[o] = -1;
                a.path_slot[o] = -1;
            }
            continue;
        }
        int js;
        float q;
        if (greedy) {
            const uint32_t at = __ballot_sync(FULL, lane < NC && v == mx);
            js = __ffs(at) - 1;
            q = lane == js ? 1.0f : 0.0f;
        } else {
            const float e = lane < NC ? expf(v - mx) : 0.0f;
            const float tot = warp_sum(e);
            float cum = e;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const float tt = __shfl_up_sync(FULL, cum, d);
                if (lane >= d) cum += tt;
            }
            const float thr = a.u_walk[o] * tot;
            const uint32_t hit = __ballot_sync(FULL, lane < NC && cum > thr);
            if (hit) {
                js = __ffs(hit) - 1;
            } else {
                const uint32_t pos = __ballot_sync(FULL, lane < NC && e > 0.0f);
                js = 31 - __clz(pos);
            }
            q = e / tot;
        }
        if (lane < NC) a.q_sel[o * NC + lane] = q;
        if (lane == 0) {
            a.path_slot[o] = js;
            a.path_tok[o] = sC[t * NC + js];
        }
        prev = js;
    }
}

template <bool BF16>
__global__ void __launch_bounds__(WALK_THREADS) k_pair_score_walk(WalkArgs a) {
    extern __shared__ float4 smem4[];
    float *smem = reinterpret_cast<float *>(smem4);
    const int D = a.D;
    const int LD = D + 4;  // padded row stride (floats)
    float *sA = smem;               // [16][LD]  A(pred) * gate
    float *sB = sA + NC * LD;       // [16][LD]  B(cand)
    float *sG = sB + NC * LD;       // [D]
    float *sU = sG + D;             // [16]
    int32_t *sCand = reinterpret_cast<int32_t *>(sU + NC);  // [16]
    int32_t *sPred = sCand + NC;                              // [16]
    float *sTile = reinterpret_cast<float *>(sPred + NC);    // [16][16]
    __shared__ int s_last;

    const int t = blockIdx.x;
    const int64_t b = blockIdx.y;
    const int K = a.K;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t pos = b * K + t;

    if (tid < NC) {
        sCand[tid] = a.cand_idx[pos * NC + tid];
        sU[tid] = a.cand_U[pos * NC + tid];
        int32_t p;
        if (t == 0)
            p = tid == 0 ? a.last_tok[b] : -2;  // -2: no predecessor
        else
            p = a.cand_idx[(pos - 1) * NC + tid];
        sPred[tid] = p;
    }
    for (int k = tid; k < D; k += WALK_THREADS) sG[k] = a.gate[pos * D + k];
    __syncthreads();

    // Gather: rows 0..15 are A(pred_i) * gate, rows 16..31 are B(cand_j).
    const int chunks = D / 4;
    for (int rr = warp; rr < 2 * NC; rr += WALK_THREADS / 32) {
        const bool isA = rr < NC;
        const int i = isA ? rr : rr - NC;
        const int32_t id = isA ? sPred[i] : sCand[i];
        const bool ok = id >= 0 && id < a.V;
        float *dst = (isA ? sA : sB) + i * LD;
        for (int c = lane; c < chunks; c += 32) {
            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (ok) load_row_chunk<BF16>(isA ? a.A : a.Bt, id, D, c * 4, v);
            if (isA) {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] *= sG[c * 4 + e];
            }
            *reinterpret_cast<float4 *>(dst + c * 4) = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
    __syncthreads();

    // 16 blocks of 4x4 outputs x 16 k-slices.  warp w holds blocks 2w, 2w+1.
    {
        const int blk = warp * 2 + (lane >> 4);
        const int ks = lane & 15;
        const int i0 = (blk >> 2) * 4;
        const int j0 = (blk & 3) * 4;
        float acc[4][4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[ii][jj] = 0.0f;
        for (int c = ks; c < chunks; c += 16) {
            float4 av[4], bv[4];
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) av[ii] = *reinterpret_cast<const float4 *>(sA + (i0 + ii) * LD + c * 4);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) bv[jj] = *reinterpret_cast<const float4 *>(sB + (j0 + jj) * LD + c * 4);
#pragma unroll
            for (int ii = 0; ii < 4; ++ii)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    float s = acc[ii][jj];
                    s = fmaf(av[ii].x, bv[jj].x, s);
                    s = fmaf(av[ii].y, bv[jj].y, s);
                    s = fmaf(av[ii].z, bv[jj].z, s);
                    s = fmaf(av[ii].w, bv[jj].w, s);
                    acc[ii][jj] = s;
                }
        }
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                float s = acc[ii][jj];
                s += __shfl_xor_sync(FULL, s, 1);
                s += __shfl_xor_sync(FULL, s, 2);
                s += __shfl_xor_sync(FULL, s, 4);
                s += __shfl_xor_sync(FULL, s, 8);
                acc[ii][jj] = s;
            }
        if (ks == 0) {
#pragma unroll
            for (int ii = 0; ii < 4; ++ii)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int i = i0 + ii, j = j0 + jj;
                    const int32_t p = sPred[i], c = sCand[j];
                    float s;
                    if (p == -2)
                        s = NEG_INF;
                    else if (p < 0 || p >= a.V || c < 0 || c >= a.V)
                        s = NAN;
                    else
                        s = sU[j] + acc[ii][jj];
                    sTile[i * NC + j] = s;
                }
        }
    }
    __syncthreads();
    a.scores[pos * NC * NC + tid] = sTile[tid];
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int old = atomicAdd(&a.tickets[b], 1);
        s_last = old == K - 1;
        if (s_last) a.tickets[b] = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // Last tile of request b: load the K tiles and candidate ids, then walk.
    float *sS = smem;                                            // [K][16][16]
    int32_t *sC = reinterpret_cast<int32_t *>(smem + K * NC * NC);  // [K][16]
    __syncthreads();
    for (int i = tid; i < K * NC * NC; i += WALK_THREADS) sS[i] = __ldcg(a.scores + b * K * NC * NC + i);
    for (int i = tid; i < K * NC; i += WALK_THREADS) sC[i] = a.cand_idx[b * K * NC + i];
    __syncthreads();
    if (warp == 0) walk_request(a, b, sS, sC, lane);
}

static size_t walk_smem(int D, int K) {
    const size_t tile = (2 * NC * (D + 4) + D + NC) * sizeof(float) + 2 * NC * sizeof(int32_t) +
                        NC * NC * sizeof(float);
    const size_t walk = static_cast<size_t>(K) * NC * NC * sizeof(float) + K * NC * sizeof(int32_t);
    return tile > walk ? tile : walk;
}

}  // namespace dfl

using namespace dfl;

extern "C" size_t dflash2_pair_score_walk_workspace_bytes(int64_t B) {
    if (B < 0) return 0;
    return static_cast<size_t>((B * sizeof(int32_t) + 255) / 256 * 256);
}

extern "C" dflash2_status dflash2_pair_score_walk(int64_t B, int32_t K, const int32_t *cand_idx,
                                                  const float *cand_U, const int32_t *last_tok,
                                                  const void *A, const void *Bt, dflash2_dtype tdt,
                                                  int64_t V, int32_t D, const float *gate,
                                                  const dflash2_sampling *params, const float *u_walk,
                                                  int32_t *path_tok, int32_t *path_slot, float *q_sel,
                                                  float *scores, void *ws, size_t ws_bytes,
                                                  dflash2_stream stream) {
    if (!dtype_ok(tdt) || B < 0 || K < 1 || K > DFLASH2_MAX_K || V < NC || V >= (int64_t(1) << 31) ||
        D < 16 || D > 1024 || (D & (D - 1)) != 0)
        return DFLASH2_ERR_INVALID_ARG;
    if (B == 0) return DFLASH2_OK;
    if (!cand_idx || !cand_U || !last_tok || !A || !Bt || !gate || !path_tok || !path_slot || !q_sel ||
        !scores || !ws || !aligned16(A) || !aligned16(Bt))
        return DFLASH2_ERR_INVALID_ARG;
    if (params && !u_walk) return DFLASH2_ERR_INVALID_ARG;
    if (ws_bytes < dflash2_pair_score_walk_workspace_bytes(B)) return DFLASH2_ERR_WORKSPACE;
    if (B > 65535) return DFLASH2_ERR_UNSUPPORTED;
    WalkArgs a;
    a.B = B;
    a.K = K;
    a.V = V;
    a.D = D;
    a.cand_idx = cand_idx;
    a.cand_U = cand_U;
    a.last_tok = last_tok;
    a.A = A;
    a.Bt = Bt;
    a.gate = gate;
    a.params = params;
    a.u_walk = u_walk;
    a.path_tok = path_tok;
    a.path_slot = path_slot;
    a.q_sel = q_sel;
    a.scores = scores;
    a.tickets = static_cast<int32_t *>(ws);
    const size_t smem = walk_smem(D, K);
    const dim3 grid(static_cast<unsigned>(K), static_cast<unsigned>(B));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t smem_max = walk_smem(1024, DFLASH2_MAX_K);
    if (tdt == DFLASH2_BF16) {
        blocks_per_sm(reinterpret_cast<const void *>(&k_pair_score_walk<true>), WALK_THREADS, smem_max);
        k_pair_score_walk<true><<<grid, WALK_THREADS, smem, s>>>(a);
    } else {
        blocks_per_sm(reinterpret_cast<const void *>(&k_pair_score_walk<false>), WALK_THREADS, smem_max);
        k_pair_score_walk<false><<<grid, WALK_THREADS, smem, s>>>(a);
    }
    return after_launch();
}

// ---------------------------------------------------------------------------
// dflash2_pair_score_walk_noalloc: the same call for callers that cannot hand
// this library any device memory of their own.  The per-request tickets live
// in a fixed array in the library's device memory instead of a workspace.
namespace dfl {

constexpr int64_t WALK_NOALLOC_MAX_B = DFLASH2_WALK_NOALLOC_MAX_B;

// One ticket per request; every GPU that loads the library holds this array
// (64 KB) until the process exits.  All calls share it.
static __device__ __align__(256) int32_t g_walk_noalloc_tickets[WALK_NOALLOC_MAX_B];

// Device address of the ticket array on the current device, looked up once
// per device with that device current.  In host code the array's name is
// only a host-side stand-in, so the address must come from the runtime.
static int32_t *walk_noalloc_tickets() {
    static int32_t *addr[64] = {nullptr};
    static std::mutex mu;
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_walk_noalloc_tickets) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<int32_t *>(p);
    }
    return addr[dev];
}

}  // namespace dfl

extern "C" dflash2_status dflash2_pair_score_walk_noalloc(
    int64_t B, int32_t K, const int32_t *cand_idx, const float *cand_U, const int32_t *last_tok, const void *A,
    const void *Bt, dflash2_dtype tdt, int64_t V, int32_t D, const float *gate, const dflash2_sampling *params,
    const float *u_walk, int32_t *path_tok, int32_t *path_slot, float *q_sel, float *scores,
    dflash2_stream stream) {
    if (B > dfl::WALK_NOALLOC_MAX_B) return DFLASH2_ERR_WORKSPACE;
    if (B <= 0)
        return dflash2_pair_score_walk(B, K, cand_idx, cand_U, last_tok, A, Bt, tdt, V, D, gate, params, u_walk,
                                       path_tok, path_slot, q_sel, scores, nullptr, 0, stream);
    int32_t *tickets = dfl::walk_noalloc_tickets();
    if (!tickets) return DFLASH2_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The tickets must start at zero: clear this call's share of the array.
    if (cudaMemsetAsync(tickets, 0, static_cast<size_t>(B) * sizeof(int32_t), s) != cudaSuccess)
        return DFLASH2_ERR_CUDA;
    return dflash2_pair_score_walk(B, K, cand_idx, cand_U, last_tok, A, Bt, tdt, V, D, gate, params, u_walk,
                                   path_tok, path_slot, q_sel, scores, tickets,
                                   sizeof(int32_t) * static_cast<size_t>(dfl::WALK_NOALLOC_MAX_B), stream);
}
