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
// score tile on the tensor cores.  It also settles, for each of the 16
// possible predecessors, the step's choice and distribution, and stores these
// tables straight into the shared memory of the first CTA of the request's
// thread-block cluster; after one cluster barrier that CTA chains them from
// the last verified token.
#include <cuda_bf16.h>

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
};

// Walk tables of one position's tile, for every predecessor row i: the row
// is dead (it holds a NaN or only -inf), the chosen slot js (greedy: the
// first maximum; sampled: the first slot whose cumulative q exceeds u, else
// the last slot with q > 0) and the walk's distribution q over the row.
// 256 threads: thread (i = tid / 16, j = tid % 16) holds S[i][j]; a row lives
// in one half-warp.  The tables go to the arrays dQ [16][16], dJs [16] and
// dDead [16] of the cluster's first CTA (addresses as in this CTA).
__device__ __forceinline__ void tile_tables(float v, bool greedy, float u, float *dQ, int32_t *dJs, int32_t *dDead,
                                            int tid) {
    const int i = tid >> 4, j = tid & 15;
    const unsigned hw = 0xffffu << (tid & 16);  // this half-warp
    float mx = v;
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, d));  // NaN-ignoring
    const bool any_nan = __ballot_sync(FULL, v != v) & hw;
    const bool dead = any_nan || mx == NEG_INF;
    int js = 0;
    float q;
    if (greedy) {
        const uint32_t at = (__ballot_sync(FULL, v == mx) & hw) >> (tid & 16);
        js = at ? __ffs(at) - 1 : 0;
        q = j == js ? 1.0f : 0.0f;
    } else {
        const float e = dead ? 0.0f : expf(v - mx);
        float tot = e;
#pragma unroll
        for (int d = 8; d >= 1; d >>= 1) tot += __shfl_xor_sync(FULL, tot, d);
        float cum = e;
#pragma unroll
        for (int d = 1; d < 16; d <<= 1) {
            const float t = __shfl_up_sync(FULL, cum, d);
            if (j >= d) cum += t;
        }
        const float thr = u * tot;
        const uint32_t hit = (__ballot_sync(FULL, cum > thr) & hw) >> (tid & 16);
        const uint32_t pos = (__ballot_sync(FULL, e > 0.0f) & hw) >> (tid & 16);
        js = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
        q = e / tot;
    }
    st_dsmem_u32(dQ + i * NC + j, __float_as_uint(dead ? NAN : q), 0);
    if (j == 0) {
        st_dsmem_u32(dJs + i, static_cast<uint32_t>(js), 0);
        st_dsmem_u32(dDead + i, dead ? 1u : 0u, 0);
    }
}

// The walk of request b (one warp) over the K positions' tables: from the
// last verified token (row 0 of position 0), each step takes the chosen slot
// of the predecessor's row; a dead row ends the walk (that step and the rest
// get token -1, slot -1 and NaN q).
__device__ void walk_request(const WalkArgs &a, int64_t b, const float *sQ, const int32_t *sJs,
                             const int32_t *sDead, const int32_t *sC, int lane) {
    const int K = a.K;
    int prev = 0;
    bool dead = false;
    for (int t = 0; t < K; ++t) {
        const int64_t o = b * K + t;
        dead = dead || sDead[t * NC + prev] != 0;
        if (dead) {
            if (lane < NC) a.q_sel[o * NC + lane] = NAN;
            if (lane == 0) {
                a.path_tok[o] = -1;
                a.path_slot[o] = -1;
            }
            continue;
        }
        const int js = sJs[t * NC + prev];
        if (lane < NC) a.q_sel[o * NC + lane] = sQ[(t * NC + prev) * NC + lane];
        if (lane == 0) {
            a.path_slot[o] = js;
            a.path_tok[o] = sC[t * NC + js];
        }
        prev = js;
    }
}

// Warp-level bf16 tensor-core product (m16n8k16, fp32 accumulation).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// x as the sum of three bf16 (each the nearest bf16 of what remains): the
// parts carry about 24 significant bits, fp32's precision.
__device__ __forceinline__ void split_bf16(float x, uint16_t &hi, uint16_t &mid, uint16_t &lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(h);
    const __nv_bfloat16 m = __float2bfloat16_rn(r1);
    const __nv_bfloat16 l = __float2bfloat16_rn(r1 - __bfloat162float(m));
    hi = __bfloat16_as_ushort(h);
    mid = __bfloat16_as_ushort(m);
    lo = __bfloat16_as_ushort(l);
}

template <bool BF16>
__global__ void __launch_bounds__(WALK_THREADS, 4) k_pair_score_walk(WalkArgs a) {
    extern __shared__ float4 smem4[];
    unsigned char *base = reinterpret_cast<unsigned char *>(smem4);
    const int D = a.D;
    const int K = a.K;
    // Operand rows.  bf16 tables: A(pred) * gate split into three bf16 parts
    // and B(cand) as stored, rows of D + 8 bf16 (the pad spreads the rows
    // over the banks); f32 tables: fp32 rows of D + 4.
    const int LDH = D + 8, LDF = D + 4;
    const size_t opbytes = BF16 ? 4 * NC * LDH * sizeof(uint16_t) : 2 * NC * LDF * sizeof(float);
    uint16_t *sAh = reinterpret_cast<uint16_t *>(base);
    uint16_t *sAm = sAh + NC * LDH;
    uint16_t *sAl = sAm + NC * LDH;
    uint16_t *sBh = sAl + NC * LDH;
    float *sAf = reinterpret_cast<float *>(base);
    float *sBf = sAf + NC * LDF;
    float *sG = reinterpret_cast<float *>(base + opbytes);  // [D]
    float *sU = sG + D;                                      // [16]
    int32_t *sCand = reinterpret_cast<int32_t *>(sU + NC);  // [16]
    int32_t *sPred = sCand + NC;                              // [16]
    float *sPart = reinterpret_cast<float *>(sPred + NC);     // [8][16][16] per-warp partial tiles
    float *sQAll = sPart + 8 * NC * NC;                         // [K][16][16] (first CTA)
    int32_t *sJsAll = reinterpret_cast<int32_t *>(sQAll + K * NC * NC);  // [K][16]
    int32_t *sDeadAll = sJsAll + K * NC;                                   // [K][16]
    int32_t *sCAll = sDeadAll + K * NC;                                    // [K][16]

    const int t = blockIdx.x;  // = rank in the request's cluster
    const int64_t b = blockIdx.y;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t pos = b * K + t;
    pdl_wait();  // the candidates and the gate come from the grids before this one

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
    if (t == 0)
        for (int i = tid; i < K * NC; i += WALK_THREADS) sCAll[i] = a.cand_idx[b * K * NC + i];
    const float T = a.params ? a.params[b].temperature : 0.0f;
    const bool greedy = !(T > 0.0f);
    const float u = greedy ? 0.0f : a.u_walk[pos];
    __syncthreads();

    // Gather: rows 0..15 are A(pred_i) * gate, rows 16..31 are B(cand_j), in
    // 16-byte chunks.  D is a power of two, so a row has cpr = 2^lcpr chunks
    // and a pass of the 256 threads covers rpp = 256 / cpr rows: thread tid
    // takes chunk tid mod cpr of rows tid / cpr + k rpp, with up to four loads
    // in flight before it uses any.
    {
        constexpr int VEPL = BF16 ? 8 : 4;  // elements per chunk
        const int lcpr = __ffs(D / VEPL) - 1;
        const int c = tid & ((1 << lcpr) - 1);
        const int rpp = WALK_THREADS >> lcpr;
        const int r0 = tid >> lcpr;
        const int npass = (2 * NC + rpp - 1) / rpp;
        for (int p0 = 0; p0 < npass; p0 += 4) {
            uint4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int rr = r0 + (p0 + k) * rpp;
                v[k] = make_uint4(0u, 0u, 0u, 0u);
                if (p0 + k < npass && rr < 2 * NC) {
                    const bool isA = rr < NC;
                    const int32_t id = isA ? sPred[rr] : sCand[rr - NC];
                    if (id >= 0 && id < a.V) {
                        const char *tab = static_cast<const char *>(isA ? a.A : a.Bt);
                        v[k] = *reinterpret_cast<const uint4 *>(tab + (static_cast<int64_t>(id) * D + c * VEPL) *
                                                                          (BF16 ? 2 : 4));
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int rr = r0 + (p0 + k) * rpp;
                if (!(p0 + k < npass && rr < 2 * NC)) continue;
                if (BF16) {
                    if (rr < NC) {
                        const uint32_t wv[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                        uint32_t ph[4], pm[4], pl[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            uint16_t h0, m0, l0, h1, m1, l1;
                            split_bf16(bf16lo(wv[e2]) * sG[c * 8 + 2 * e2], h0, m0, l0);
                            split_bf16(bf16hi(wv[e2]) * sG[c * 8 + 2 * e2 + 1], h1, m1, l1);
                            ph[e2] = h0 | (static_cast<uint32_t>(h1) << 16);
                            pm[e2] = m0 | (static_cast<uint32_t>(m1) << 16);
                            pl[e2] = l0 | (static_cast<uint32_t>(l1) << 16);
                        }
                        *reinterpret_cast<uint4 *>(sAh + rr * LDH + c * 8) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                        *reinterpret_cast<uint4 *>(sAm + rr * LDH + c * 8) = make_uint4(pm[0], pm[1], pm[2], pm[3]);
                        *reinterpret_cast<uint4 *>(sAl + rr * LDH + c * 8) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
                    } else {
                        *reinterpret_cast<uint4 *>(sBh + (rr - NC) * LDH + c * 8) = v[k];  // exact
                    }
                } else {
                    float4 f = make_float4(__uint_as_float(v[k].x), __uint_as_float(v[k].y),
                                           __uint_as_float(v[k].z), __uint_as_float(v[k].w));
                    if (rr < NC) {
                        f.x *= sG[c * 4];
                        f.y *= sG[c * 4 + 1];
                        f.z *= sG[c * 4 + 2];
                        f.w *= sG[c * 4 + 3];
                    }
                    *reinterpret_cast<float4 *>((rr < NC ? sAf + rr * LDF : sBf + (rr - NC) * LDF) + c * 4) = f;
                }
            }
        }
    }
    __syncthreads();

    // The 16 x 16 dot products.  bf16: warp w takes k-steps w, w + 8, ... of
    // 16 and both 8-column halves, on the tensor cores (the three parts of
    // A, smallest first); the eight partial tiles are summed in warp order.  f32: one thread
    // per score with fp32 FMAs.
    float dot;
    if (BF16) {
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int gid = lane >> 2, tig = lane & 3;
        for (int ks = warp; ks < D / 16; ks += 8) {
            const int k0 = ks * 16 + tig * 2;
            uint32_t ah[4], am[4], al[4];
            am[0] = *reinterpret_cast<const uint32_t *>(sAm + gid * LDH + k0);
            am[1] = *reinterpret_cast<const uint32_t *>(sAm + (gid + 8) * LDH + k0);
            am[2] = *reinterpret_cast<const uint32_t *>(sAm + gid * LDH + k0 + 8);
            am[3] = *reinterpret_cast<const uint32_t *>(sAm + (gid + 8) * LDH + k0 + 8);
            ah[0] = *reinterpret_cast<const uint32_t *>(sAh + gid * LDH + k0);
            ah[1] = *reinterpret_cast<const uint32_t *>(sAh + (gid + 8) * LDH + k0);
            ah[2] = *reinterpret_cast<const uint32_t *>(sAh + gid * LDH + k0 + 8);
            ah[3] = *reinterpret_cast<const uint32_t *>(sAh + (gid + 8) * LDH + k0 + 8);
            al[0] = *reinterpret_cast<const uint32_t *>(sAl + gid * LDH + k0);
            al[1] = *reinterpret_cast<const uint32_t *>(sAl + (gid + 8) * LDH + k0);
            al[2] = *reinterpret_cast<const uint32_t *>(sAl + gid * LDH + k0 + 8);
            al[3] = *reinterpret_cast<const uint32_t *>(sAl + (gid + 8) * LDH + k0 + 8);
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
                const uint16_t *br = sBh + (nb * 8 + gid) * LDH + k0;
                const uint32_t b0 = *reinterpret_cast<const uint32_t *>(br);
                const uint32_t b1 = *reinterpret_cast<const uint32_t *>(br + 8);
                mma_bf16_16816(acc[nb], al, b0, b1);  // smallest parts first
                mma_bf16_16816(acc[nb], am, b0, b1);
                mma_bf16_16816(acc[nb], ah, b0, b1);
            }
        }
        // fragment (row gid / gid + 8, columns nb*8 + tig*2 + {0,1}) -> partial tile
        float *pw = sPart + warp * NC * NC;
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
            const int c = nb * 8 + tig * 2;
            *reinterpret_cast<float2 *>(pw + gid * NC + c) = make_float2(acc[nb][0], acc[nb][1]);
            *reinterpret_cast<float2 *>(pw + (gid + 8) * NC + c) = make_float2(acc[nb][2], acc[nb][3]);
        }
        __syncthreads();
        dot = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) dot += sPart[w * NC * NC + tid];
    } else {
        const int i = tid >> 4, j = tid & 15;
        const float *ar = sAf + i * LDF;
        const float *br = sBf + j * LDF;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int c = 0; c < D / 4; ++c) {
            const float4 x = *reinterpret_cast<const float4 *>(ar + c * 4);
            const float4 y = *reinterpret_cast<const float4 *>(br + c * 4);
            acc[0] = fmaf(x.x, y.x, acc[0]);
            acc[1] = fmaf(x.y, y.y, acc[1]);
            acc[2] = fmaf(x.z, y.z, acc[2]);
            acc[3] = fmaf(x.w, y.w, acc[3]);
        }
        dot = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    float s;
    {
        const int i = tid >> 4, j = tid & 15;
        const int32_t p = sPred[i], c = sCand[j];
        if (p == -2)
            s = NEG_INF;
        else if (p < 0 || p >= a.V || c < 0 || c >= a.V)
            s = NAN;
        else
            s = sU[j] + dot;
    }
    tile_tables(s, greedy, u, sQAll + t * NC * NC, sJsAll + t * NC, sDeadAll + t * NC, tid);
    a.scores[pos * NC * NC + tid] = s;
    // Every position's tables are in the first CTA once all have arrived
    // (release / acquire); nothing reads another CTA's memory after this.
    cluster_sync();
    // The next grid (it waits for this one to complete before it reads
    // anything) is scheduled only now: its CTAs then find the SMs free all
    // at once.  Scheduled while this grid still held the SMs, some of them
    // could start only when others of its own CTAs finished.
    pdl_trigger();
    if (t == 0 && warp == 0) walk_request(a, b, sQAll, sJsAll, sDeadAll, sCAll, lane);
}

static size_t walk_smem(int D, int K) {
    const size_t ops = 4 * NC * (D + 8) * sizeof(uint16_t) > 2 * NC * (D + 4) * sizeof(float)
                           ? 4 * NC * (D + 8) * sizeof(uint16_t)
                           : 2 * NC * (D + 4) * sizeof(float);
    return ops + (D + NC) * sizeof(float) + 2 * NC * sizeof(int32_t) + 8 * NC * NC * sizeof(float) +
           static_cast<size_t>(K) * (NC * NC * sizeof(float) + 3 * NC * sizeof(int32_t));
}

// Whether a cluster of K CTAs with the walk's shared memory at D fits on this
// GPU at all (cudaOccupancyMaxActiveClusters > 0).  Clusters above the
// portable 8 must fit in one GPC, so a large K at a large D might not.
// Cached per device and (K, D).
static bool walk_cluster_fits(const void *fn, const cudaLaunchConfig_t &cfg, int K, int D) {
    static signed char fits[64][DFLASH2_MAX_K + 1][7];  // 0 unknown, 1 fits, -1 does not
    static std::mutex mu;
    const int dev = current_device();
    int di = 0;
    while ((16 << di) < D) ++di;  // D = 16 << di, di in 0..6
    std::lock_guard<std::mutex> lock(mu);
    signed char *f = (dev >= 0 && dev < 64) ? &fits[dev][K][di] : nullptr;
    if (f && *f) return *f > 0;
    int n = 0;
    const bool ok = cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess && n > 0;
    if (!ok) cudaGetLastError();  // a refused query is an answer here, not a sticky launch error
    if (f) *f = ok ? 1 : -1;
    return ok;
}

// Launch one cluster of K CTAs per request (K up to 15: clusters above the
// portable 8 are allowed on this GPU once the kernel opts in).  UNSUPPORTED
// when such a cluster cannot be resident at this D.
template <bool BF16>
static dflash2_status launch_walk(const WalkArgs &a, cudaStream_t s) {
    const void *fn = reinterpret_cast<const void *>(&k_pair_score_walk<BF16>);
    static int opted[64] = {0};
    static std::mutex mu;
    {
        const int dev = current_device();
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 0 && dev < 64 && !opted[dev]) {
            cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            opted[dev] = 1;
        }
    }
    blocks_per_sm(fn, WALK_THREADS, walk_smem(1024, DFLASH2_MAX_K));  // raises the shared-memory limit once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.K), static_cast<unsigned>(a.B), 1);
    cfg.blockDim = dim3(WALK_THREADS, 1, 1);
    cfg.dynamicSmemBytes = walk_smem(a.D, a.K);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.K);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
    if (!walk_cluster_fits(fn, cfg, a.K, a.D)) return DFLASH2_ERR_UNSUPPORTED;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, k_pair_score_walk<BF16>, a) != cudaSuccess) return DFLASH2_ERR_CUDA;
    return after_launch();
}

}  // namespace dfl

using namespace dfl;

extern "C" dflash2_status dflash2_pair_score_walk(int64_t B, int32_t K, const int32_t *cand_idx,
                                                  const float *cand_U, const int32_t *last_tok,
                                                  const void *A, const void *Bt, dflash2_dtype tdt,
                                                  int64_t V, int32_t D, const float *gate,
                                                  const dflash2_sampling *params, const float *u_walk,
                                                  int32_t *path_tok, int32_t *path_slot, float *q_sel,
                                                  float *scores, dflash2_stream stream) {
    if (!dtype_ok(tdt) || B < 0 || K < 1 || K > DFLASH2_MAX_K || V < NC || V >= (int64_t(1) << 31) ||
        D < 16 || D > 1024 || (D & (D - 1)) != 0)
        return DFLASH2_ERR_INVALID_ARG;
    if (B == 0) return DFLASH2_OK;
    if (!cand_idx || !cand_U || !last_tok || !A || !Bt || !gate || !path_tok || !path_slot || !q_sel ||
        !scores || !aligned16(A) || !aligned16(Bt))
        return DFLASH2_ERR_INVALID_ARG;
    if (params && !u_walk) return DFLASH2_ERR_INVALID_ARG;
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
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return tdt == DFLASH2_BF16 ? launch_walk<true>(a, s) : launch_walk<false>(a, s);
}
