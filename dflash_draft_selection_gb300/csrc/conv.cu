// conv.cu -- dflash2_conv2tap: the drafter's two-tap dynamic depthwise
// convolution.
//
// DFlash 2 proposer issue, "What upstream shipped" item 2:
// Conv(x)_t = k_{t,0} * x_t + k_{t,1} * x_{t-1}, the first position tapping the
// last verified token's hidden state; FreeToken PR 857, "Details"/Refused at
// startup (conv_group_size divides the hidden size): with group size G, G
// adjacent channels share one tap pair.
//
// An elementwise stream.  bf16 outputs are the exact value of the
// two products' sum rounded once to bf16: both products of bf16 operands are
// exact in fp32, their fp32 sum s is corrected by the two-sum error e only
// when s lies exactly on a bf16 rounding midpoint.
#include "common.cuh"
#include "host.hpp"

namespace dfl {

constexpr int CONV_THREADS = 256;

__device__ __forceinline__ unsigned short round_pair_bf16(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    const uint32_t u = __float_as_uint(s);
    if (s != s) return 0x7fc0;
    const uint32_t low = u & 0xffffu;
    uint32_t r = u >> 16;
    if (low == 0x8000u && e != 0.0f) {
        // exactly on a midpoint of s's bf16 neighbours: the exact value is on e's side
        if ((e > 0.0f) == (s > 0.0f)) r += 1;
    } else if (low > 0x8000u || (low == 0x8000u && (r & 1u))) {
        r += 1;
    }
    return static_cast<unsigned short>(r);
}

struct ConvArgs {
    const void *x, *k0, *k1, *x_prev;
    void *y;
    int64_t B, H;
    int T, G;
};

__device__ __forceinline__ float ldbf(const void *p, int64_t i) {
    return __uint_as_float(static_cast<uint32_t>(static_cast<const unsigned short *>(p)[i]) << 16);
}

// bf16, one tap pair per channel, H a multiple of 8: 16-byte vectors.  The
// grid's y dimension walks the tokens (b, t) and x the token's channel
// vectors, so a token's indices are computed once, not per vector.
__global__ void __launch_bounds__(CONV_THREADS) k_conv_bf16_vec(ConvArgs a) {
    const int64_t tokens = a.B * a.T;
    const int64_t hv = a.H / 8;
    for (int64_t bt = blockIdx.y; bt < tokens; bt += gridDim.y) {
        const int t = static_cast<int>(bt % a.T);
        const int64_t b = bt / a.T;
        const unsigned short *xr = static_cast<const unsigned short *>(a.x) + bt * a.H;
        const unsigned short *pr = t == 0 ? static_cast<const unsigned short *>(a.x_prev) + b * a.H : xr - a.H;
        const unsigned short *k0r = static_cast<const unsigned short *>(a.k0) + bt * a.H;
        const unsigned short *k1r = static_cast<const unsigned short *>(a.k1) + bt * a.H;
        unsigned short *yr = static_cast<unsigned short *>(a.y) + bt * a.H;
        for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < hv;
             v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(xr + v * 8);
            const uint4 pv = *reinterpret_cast<const uint4 *>(pr + v * 8);
            const uint4 k0v = *reinterpret_cast<const uint4 *>(k0r + v * 8);
            const uint4 k1v = *reinterpret_cast<const uint4 *>(k1r + v * 8);
            const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
            const uint32_t ps[4] = {pv.x, pv.y, pv.z, pv.w};
            const uint32_t k0s[4] = {k0v.x, k0v.y, k0v.z, k0v.w};
            const uint32_t k1s[4] = {k1v.x, k1v.y, k1v.z, k1v.w};
            uint32_t out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const unsigned short lo =
                    round_pair_bf16(bf16lo(k0s[i]) * bf16lo(xs[i]), bf16lo(k1s[i]) * bf16lo(ps[i]));
                const unsigned short hi =
                    round_pair_bf16(bf16hi(k0s[i]) * bf16hi(xs[i]), bf16hi(k1s[i]) * bf16hi(ps[i]));
                out[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            *reinterpret_cast<uint4 *>(yr + v * 8) = make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
}

// Any shape / group size: one element per step.
template <bool BF16>
__global__ void __launch_bounds__(CONV_THREADS) k_conv_scalar(ConvArgs a) {
    const int64_t n = a.B * a.T * a.H;
    const int64_t Hk = a.H / a.G;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t bt = e / a.H;
        const int64_t c = e - bt * a.H;
        const int t = static_cast<int>(bt % a.T);
        const int64_t b = bt / a.T;
        const int64_t ko = bt * Hk + c / a.G;
        const int64_t po = t == 0 ? b * a.H + c : e - a.H;
        const void *psrc = t == 0 ? a.x_prev : a.x;
        if (BF16) {
            const float p0 = ldbf(a.k0, ko) * ldbf(a.x, e);
            const float p1 = ldbf(a.k1, ko) * ldbf(psrc, po);
            static_cast<unsigned short *>(a.y)[e] = round_pair_bf16(p0, p1);
        } else {
            const float *x = static_cast<const float *>(a.x);
            const float *xp = static_cast<const float *>(psrc);
            const float k0 = static_cast<const float *>(a.k0)[ko];
            const float k1 = static_cast<const float *>(a.k1)[ko];
            static_cast<float *>(a.y)[e] = fmaf(k0, x[e], k1 * xp[po]);
        }
    }
}

// -------------------------------------------------- grouped dynamic taps --
// The taps of dflash2_dynconv2tap: k0 = taps[bt, c / G] (f32, from the
// gate GEMM), k1 = 1 - k0; y = fma(k0, x_t, k1 x_{t-1}) in fp32, rounded
// once to bf16 for bf16 outputs.
struct DynArgs {
    const void *x, *x_prev;
    const float *taps;
    void *y;
    int64_t B, H;
    int T, G;
};

__device__ __forceinline__ uint32_t f32_to_bf16_rn(float v) {
    const uint32_t u = __float_as_uint(v);
    if (v != v) return 0x7fc0u;
    return (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
}

// bf16 with H and G multiples of 8: 16-byte vectors, one tap per vector.
__global__ void __launch_bounds__(CONV_THREADS) k_dynconv_bf16_vec(DynArgs a) {
    const int64_t tokens = a.B * a.T;
    const int64_t hv = a.H / 8;
    const int64_t Hk = a.H / a.G;
    for (int64_t bt = blockIdx.y; bt < tokens; bt += gridDim.y) {
        const int t = static_cast<int>(bt % a.T);
        const int64_t b = bt / a.T;
        const unsigned short *xr = static_cast<const unsigned short *>(a.x) + bt * a.H;
        const unsigned short *pr = t == 0 ? static_cast<const unsigned short *>(a.x_prev) + b * a.H : xr - a.H;
        const float *kr = a.taps + bt * Hk;
        unsigned short *yr = static_cast<unsigned short *>(a.y) + bt * a.H;
        for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < hv;
             v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const float k0 = kr[v * 8 / a.G], k1 = 1.0f - k0;
            const uint4 xv = *reinterpret_cast<const uint4 *>(xr + v * 8);
            const uint4 pv = *reinterpret_cast<const uint4 *>(pr + v * 8);
            const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
            const uint32_t ps[4] = {pv.x, pv.y, pv.z, pv.w};
            uint32_t out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = f32_to_bf16_rn(fmaf(k0, bf16lo(xs[i]), k1 * bf16lo(ps[i])));
                const uint32_t hi = f32_to_bf16_rn(fmaf(k0, bf16hi(xs[i]), k1 * bf16hi(ps[i])));
                out[i] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4 *>(yr + v * 8) = make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
}

// Any shape: one element per step.
template <bool BF16>
__global__ void __launch_bounds__(CONV_THREADS) k_dynconv_scalar(DynArgs a) {
    const int64_t n = a.B * a.T * a.H;
    const int64_t Hk = a.H / a.G;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t bt = e / a.H;
        const int64_t c = e - bt * a.H;
        const int t = static_cast<int>(bt % a.T);
        const int64_t b = bt / a.T;
        const float k0 = a.taps[bt * Hk + c / a.G], k1 = 1.0f - k0;
        const int64_t po = t == 0 ? b * a.H + c : e - a.H;
        const void *psrc = t == 0 ? a.x_prev : a.x;
        if (BF16) {
            const float v = fmaf(k0, ldbf(a.x, e), k1 * ldbf(psrc, po));
            static_cast<unsigned short *>(a.y)[e] = static_cast<unsigned short>(f32_to_bf16_rn(v));
        } else {
            const float *x = static_cast<const float *>(a.x);
            const float *xp = static_cast<const float *>(psrc);
            static_cast<float *>(a.y)[e] = fmaf(k0, x[e], k1 * xp[po]);
        }
    }
}

}  // namespace dfl

using namespace dfl;

extern "C" dflash2_status dflash2_dynconv2tap(const void *x, const void *x_prev, const void *Wd, dflash2_dtype dt,
                                              int64_t B, int32_t T, int64_t H, int32_t group_size, float *taps,
                                              void *y, dflash2_stream stream) {
    if (!dtype_ok(dt) || B < 0 || T < 1 || H < 1 || group_size < 1 || H % group_size != 0)
        return DFLASH2_ERR_INVALID_ARG;
    if (B == 0) return DFLASH2_OK;
    if (!x || !x_prev || !Wd || !taps || !y || !aligned16(x) || !aligned16(Wd) || !aligned16(taps))
        return DFLASH2_ERR_INVALID_ARG;
    const int64_t Hk = H / group_size;
    if (dt == DFLASH2_BF16 && (H % 64 != 0 || Hk < 16 || Hk > 512 || (Hk & (Hk - 1)) != 0))
        return DFLASH2_ERR_UNSUPPORTED;  // the tensor-core taps' tiles
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // x is typically the previous kernel's output: the projection starts after it completes
    const dflash2_status st = gate_launch(x, dt, B * T, H, Wd, static_cast<int>(Hk), taps, s, false);
    if (st != DFLASH2_OK) return st;
    DynArgs a{x, x_prev, taps, y, B, H, T, group_size};
    const bool vec = dt == DFLASH2_BF16 && H % 8 == 0 && group_size % 8 == 0 && aligned16(x_prev) && aligned16(y);
    if (vec) {
        const int64_t tokens = B * T;
        const int64_t xb = (H / 8 + CONV_THREADS - 1) / CONV_THREADS;
        const int64_t yb = tokens < 65535 ? tokens : 65535;
        k_dynconv_bf16_vec<<<dim3(static_cast<unsigned>(xb), static_cast<unsigned>(yb)), CONV_THREADS, 0, s>>>(a);
    } else {
        int64_t blocks = (B * T * H + CONV_THREADS - 1) / CONV_THREADS;
        const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
        if (blocks > cap) blocks = cap;
        if (dt == DFLASH2_BF16)
            k_dynconv_scalar<true><<<static_cast<unsigned>(blocks), CONV_THREADS, 0, s>>>(a);
        else
            k_dynconv_scalar<false><<<static_cast<unsigned>(blocks), CONV_THREADS, 0, s>>>(a);
    }
    return after_launch();
}

extern "C" dflash2_status dflash2_conv2tap(const void *x, const void *k0, const void *k1,
                                           const void *x_prev, dflash2_dtype dt, int64_t B, int32_t T,
                                           int64_t H, int32_t group_size, void *y,
                                           dflash2_stream stream) {
    if (!dtype_ok(dt) || B < 0 || T < 1 || H < 1 || group_size < 1 || H % group_size != 0)
        return DFLASH2_ERR_INVALID_ARG;
    if (B == 0) return DFLASH2_OK;
    if (!x || !k0 || !k1 || !x_prev || !y) return DFLASH2_ERR_INVALID_ARG;
    ConvArgs a{x, k0, k1, x_prev, y, B, H, T, group_size};
    const int64_t n = B * T * H;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool vec = dt == DFLASH2_BF16 && group_size == 1 && H % 8 == 0 && aligned16(x) &&
                     aligned16(k0) && aligned16(k1) && aligned16(x_prev) && aligned16(y);
    if (vec) {
        const int64_t tokens = B * T;
        const int64_t xb = (H / 8 + CONV_THREADS - 1) / CONV_THREADS;
        const int64_t yb = tokens < 65535 ? tokens : 65535;
        k_conv_bf16_vec<<<dim3(static_cast<unsigned>(xb), static_cast<unsigned>(yb)), CONV_THREADS, 0, s>>>(a);
    } else {
        int64_t blocks = (n + CONV_THREADS - 1) / CONV_THREADS;
        if (blocks > cap) blocks = cap;
        if (dt == DFLASH2_BF16)
            k_conv_scalar<true><<<static_cast<unsigned>(blocks), CONV_THREADS, 0, s>>>(a);
        else
            k_conv_scalar<false><<<static_cast<unsigned>(blocks), CONV_THREADS, 0, s>>>(a);
    }
    return after_launch();
}
