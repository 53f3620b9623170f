// gate.cu -- dflash2_ctx_gate: the context gate H(h) = sigmoid(W_g h).
//
// DFlash 2 proposer issue, "What upstream shipped" item 1: the pair score is
// a low-rank bilinear attention whose 256-dim factors are scaled by a context
// gate of the drafter's hidden state; the gate is read as sigmoid(W_g h) with
// W_g: hidden -> 256 and no bias.
//
// bf16 path, the one dense contraction of the selector: a 5th-generation
// tensor-core GEMM.  gate[n, D] = sigmoid(h[n, hidden] . W_g[D, hidden]^T),
// both operands K-major.  A CTA owns a 128 x BN output tile and a slice of the
// hidden (K) dimension: TMA (cp.async.bulk.tensor, 128-byte swizzle) stages
// 128x64 and BNx64 bf16 tiles through a 3-deep mbarrier ring, one thread
// issues tcgen05.mma (kind::f16, fp32 accumulation in tensor memory), and
// tcgen05.commit releases each stage.  The ks CTAs (up to 8) of one tile
// form a thread-block cluster along K: each reads its fp32 accumulator out of tensor memory
// into shared memory, and after a cluster barrier each reduces 128/ks rows of
// the tile across the cluster's shared memories (DSMEM, fixed order, so the
// result does not depend on timing), applies the sigmoid and stores.
// f32 path: a plain CUDA-core dot product per output (small shapes).
#include "common.cuh"
#include "host.hpp"
#include "tc.cuh"

namespace dfl {

static __device__ unsigned int g_err_gate;

constexpr int GBM = 128;       // tile rows = tensor-memory lanes
constexpr int GBK = 64;        // hidden elements per stage: one 128-byte swizzle row
constexpr int GSTAGES = 3;  // small enough to share an SM with two row-scan CTAs
constexpr int GATE_THREADS = 128;
constexpr int MAX_KSPLIT = 8;  // CTAs of one tile's split-K cluster (16 measured slower)

template <int BN>
struct GateSmem {
    alignas(1024) unsigned char a[GSTAGES][GBM * GBK * 2];
    alignas(1024) unsigned char b[GSTAGES][BN * GBK * 2];
    uint64_t full[GSTAGES];
    uint64_t empty[GSTAGES];
    uint64_t accum;
    uint32_t tmem_base;
    int abort_flag;
    int issued;
};

// Instruction descriptor, kind::f16: bf16 x bf16 -> fp32, both K-major.
template <int BN>
__host__ __device__ constexpr uint32_t gate_idesc() {
    return (1u << 4)                               // D: fp32
           | (1u << 7)                             // A: bf16
           | (1u << 10)                            // B: bf16
           | (static_cast<uint32_t>(BN >> 3) << 17)  // N / 8
           | (static_cast<uint32_t>(GBM >> 4) << 24); // M / 16
}

template <int BN>
__global__ void __launch_bounds__(GATE_THREADS) k_gate_tc(const __grid_constant__ CUtensorMap tm_h,
                                                          const __grid_constant__ CUtensorMap tm_w,
                                                          float *gate, int64_t n, int D, int kblocks, int ks) {
    extern __shared__ unsigned char raw[];
    GateSmem<BN> &sm = *reinterpret_cast<GateSmem<BN> *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr uint32_t TCOLS = BN < 32 ? 32 : BN;
    constexpr int LDP = BN + 4;  // partial-tile row stride (floats)
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int mt = blockIdx.x, nt = blockIdx.y;
    const uint32_t rank = cluster_rank();
    const int kb0 = static_cast<int>((static_cast<int64_t>(kblocks) * rank) / ks);
    const int kb1 = static_cast<int>((static_cast<int64_t>(kblocks) * (rank + 1)) / ks);
    const int nkb = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < GSTAGES; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.accum, 1);
        sm.abort_flag = 0;
        sm.issued = 0;
        fence_barrier_init();
    }
    __syncwarp();
    if (warp == 1) tmem_alloc(&sm.tmem_base, TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    // The next grid may be scheduled once every CTA of this one is here; it
    // waits for this grid to complete before it reads anything.
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        // TMA producer
        int i = 0;
        for (; i < nkb; ++i) {
            const int s = i % GSTAGES;
            if (i >= GSTAGES && !mbar_wait(&sm.empty[s], ((i / GSTAGES) & 1) ^ 1)) {
                atomicOr(&g_err_gate, ERR_WAIT_TIMEOUT);
                *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
                break;
            }
            mbar_arrive_expect_tx(&sm.full[s], (GBM + BN) * GBK * 2);
            tma_load_2d(sm.a[s], &tm_h, (kb0 + i) * GBK, mt * GBM, &sm.full[s]);
            tma_load_2d(sm.b[s], &tm_w, (kb0 + i) * GBK, nt * BN, &sm.full[s]);
        }
        sm.issued = i;
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        constexpr uint32_t idesc = gate_idesc<BN>();
        for (int i = 0; i < nkb; ++i) {
            const int s = i % GSTAGES;
            const bool quick = *reinterpret_cast<volatile int *>(&sm.abort_flag) != 0;
            if (!mbar_wait(&sm.full[s], (i / GSTAGES) & 1, quick ? 0 : 4000000000ll)) {
                atomicOr(&g_err_gate, ERR_WAIT_TIMEOUT);
                *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
                break;
            }
            tc_fence_after();
            const uint64_t ad = sw128_desc(sm.a[s]);
            const uint64_t bd = sw128_desc(sm.b[s]);
#pragma unroll
            for (int k = 0; k < GBK / 16; ++k)  // 16 bf16 = 32 bytes per MMA: +2 in the address field
                mma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, i > 0 || k > 0);
            mma_commit(&sm.empty[s]);
        }
        mma_commit(&sm.accum);
    }
    __syncwarp();

    // Epilogue: tensor memory -> shared partial tile.
    const bool ok = mbar_wait(&sm.accum, 0) && *reinterpret_cast<volatile int *>(&sm.abort_flag) == 0;
    __syncwarp();  // tcgen05.ld below is warp-aligned
    tc_fence_after();
    float *part = reinterpret_cast<float *>(&sm.a[0][0]);
    const int row = warp * 32 + lane;
    // All of the warp's column blocks are loaded before one wait.
    uint32_t bits[BN];
#pragma unroll
    for (int c0 = 0; c0 < BN; c0 += 16) tmem_ld16_nowait(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, bits + c0);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < BN; i += 4) {
        float4 q = ok ? make_float4(__uint_as_float(bits[i]), __uint_as_float(bits[i + 1]), __uint_as_float(bits[i + 2]),
                                    __uint_as_float(bits[i + 3]))
                      : make_float4(NAN, NAN, NAN, NAN);
        *reinterpret_cast<float4 *>(part + row * LDP + i) = q;
    }
    if (!ok && threadIdx.x == 0) atomicOr(&g_err_gate, ERR_WAIT_TIMEOUT);
    tc_fence_before();
    cluster_sync();

    // Split-K reduction across the cluster: this CTA finishes rows
    // [rank * 128/ks, (rank+1) * 128/ks) of the tile.
    const int rows_per = GBM / ks;
    const int nvec = rows_per * BN / 4;
    for (int e = threadIdx.x; e < nvec; e += GATE_THREADS) {
        const int r = static_cast<int>(rank) * rows_per + (e * 4) / BN;
        const int c = (e * 4) % BN;
        // all partial tiles' loads first, then the sum in rank order
        float4 pv[MAX_KSPLIT];
#pragma unroll
        for (int q = 0; q < MAX_KSPLIT; ++q)
            if (q < ks) pv[q] = ld_dsmem_f4(part + r * LDP + c, static_cast<uint32_t>(q));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < MAX_KSPLIT; ++q) {
            if (q < ks) {
                acc.x += pv[q].x;
                acc.y += pv[q].y;
                acc.z += pv[q].z;
                acc.w += pv[q].w;
            }
        }
        const int64_t gr = static_cast<int64_t>(mt) * GBM + r;
        if (gr < n) {
            float4 g;
            g.x = 1.0f / (1.0f + expf(-acc.x));
            g.y = 1.0f / (1.0f + expf(-acc.y));
            g.z = 1.0f / (1.0f + expf(-acc.z));
            g.w = 1.0f / (1.0f + expf(-acc.w));
            *reinterpret_cast<float4 *>(gate + gr * D + static_cast<int64_t>(nt) * BN + c) = g;
        }
    }
    cluster_sync();
    // Do not leave copies in flight into this CTA's shared memory.
    if (threadIdx.x == 0) {
        const int issued = sm.issued;
        for (int i = issued > GSTAGES ? issued - GSTAGES : 0; i < issued; ++i)
            mbar_wait(&sm.full[i % GSTAGES], (i / GSTAGES) & 1, 200000000ll);
    }
    __syncthreads();
    tc_fence_after();
    __syncwarp();
    if (warp == 1) tmem_dealloc(tmem, TCOLS);
    // The gate reads nothing the grid before it writes, so it may run beside
    // that grid (programmatic launch); it completes only after that grid, so
    // the grids after it see both results.
    pdl_wait();
}

// f32: one warp per output element.
__global__ void __launch_bounds__(256) k_gate_f32(const float *h, const float *W, float *gate, int64_t n,
                                                  int64_t hidden, int D) {
    const int lane = threadIdx.x & 31;
    const int64_t o = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (o >= n * D) return;
    const int64_t i = o / D;
    const int k = static_cast<int>(o % D);
    float acc = 0.0f;
    for (int64_t c = lane; c < hidden; c += 32) acc = fmaf(W[k * hidden + c], h[i * hidden + c], acc);
    acc = warp_sum(acc);
    if (lane == 0) gate[o] = 1.0f / (1.0f + expf(-acc));
}

// ------------------------------------------------------------------ host ----
template <int BN>
static dflash2_status launch_gate_tc(const void *h, int64_t n, int64_t hidden, const void *Wg, int D, float *gate,
                                     cudaStream_t stream, bool early) {
    CUtensorMap tm_h, tm_w;
    if (!make_map_k64(&tm_h, h, static_cast<uint64_t>(hidden), static_cast<uint64_t>(n), GBM) ||
        !make_map_k64(&tm_w, Wg, static_cast<uint64_t>(hidden), static_cast<uint64_t>(D), BN))
        return DFLASH2_ERR_CUDA;
    const int mtiles = static_cast<int>((n + GBM - 1) / GBM);
    const int ntiles = D / BN;
    const int kblocks = static_cast<int>(hidden / GBK);
    const int64_t tiles = static_cast<int64_t>(mtiles) * ntiles;
    // Split K until the CTAs fill two per SM (clusters of up to 16).
    int ks = 1;
    while (ks < MAX_KSPLIT && tiles * ks * 2 <= 2 * static_cast<int64_t>(sm_count()) && ks * 2 <= kblocks &&
           GBM % (ks * 2) == 0)
        ks *= 2;
    const size_t smem = sizeof(GateSmem<BN>) + 1024;
    const void *fn = reinterpret_cast<const void *>(&k_gate_tc<BN>);
    {
        static int opted[64] = {0};
        static std::mutex mu;
        const int dev = current_device();
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 0 && dev < 64 && !opted[dev]) {
            cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            opted[dev] = 1;
        }
    }
    blocks_per_sm(fn, GATE_THREADS, smem);  // raises the shared-memory limit once per device
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(mtiles), static_cast<unsigned>(ntiles), static_cast<unsigned>(ks));
    cfg.blockDim = dim3(GATE_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = static_cast<unsigned>(ks);
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = early ? 2 : 1;  // without it the grid starts after the previous one completes
    if (cudaLaunchKernelEx(&cfg, k_gate_tc<BN>, tm_h, tm_w, gate, n, D, kblocks, ks) != cudaSuccess)
        return DFLASH2_ERR_CUDA;
    return after_launch();
}

unsigned int read_error_gate(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_err_gate, sizeof v);
    if (clear) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_err_gate, &z, sizeof z);
    }
    return v;
}

}  // namespace dfl

using namespace dfl;

namespace dfl {

// gate = sigmoid(h . Wg^T) for checked arguments: bf16 on the tensor cores (D a
// power of two in 16..512, hidden a multiple of 64), f32 on the CUDA cores (any D).
// With `early` the tensor-core grid may start while the previous grid runs
// (programmatic dependent launch): h and Wg must not be written by it.
dflash2_status gate_launch(const void *h, dflash2_dtype dt, int64_t n, int64_t hidden, const void *Wg, int D,
                           float *gate, cudaStream_t s, bool early) {
    if (dt == DFLASH2_F32) {
        const int64_t warps = n * D;
        const int64_t blocks = (warps * 32 + 255) / 256;
        if (blocks > 0x7fffffff) return DFLASH2_ERR_UNSUPPORTED;
        k_gate_f32<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const float *>(h),
                                                                 static_cast<const float *>(Wg), gate, n, hidden, D);
        return after_launch();
    }
    if (n >= (int64_t(1) << 31)) return DFLASH2_ERR_UNSUPPORTED;
    if (D == 16) return launch_gate_tc<16>(h, n, hidden, Wg, D, gate, s, early);
    if (D == 32) return launch_gate_tc<32>(h, n, hidden, Wg, D, gate, s, early);
    return launch_gate_tc<64>(h, n, hidden, Wg, D, gate, s, early);
}

}  // namespace dfl

extern "C" dflash2_status dflash2_ctx_gate(const void *h, dflash2_dtype dt, int64_t n, int64_t hidden,
                                           const void *Wg, int32_t D, float *gate, dflash2_stream stream) {
    if (!dtype_ok(dt) || n < 0 || hidden < 1 || D < 16 || D > 512 || (D & (D - 1)) != 0)
        return DFLASH2_ERR_INVALID_ARG;
    if (dt == DFLASH2_BF16 && hidden % GBK != 0) return DFLASH2_ERR_INVALID_ARG;
    if (n == 0) return DFLASH2_OK;
    if (!h || !Wg || !gate || !aligned16(h) || !aligned16(Wg) || !aligned16(gate)) return DFLASH2_ERR_INVALID_ARG;
    return gate_launch(h, dt, n, hidden, Wg, D, gate, reinterpret_cast<cudaStream_t>(stream), true);
}
