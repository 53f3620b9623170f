// common.cuh -- device helpers shared by the DFlash 2 kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash2.h"

namespace dfl {

constexpr int NC = DFLASH2_NC;
constexpr unsigned FULL = 0xffffffffu;
constexpr float NEG_INF = -__builtin_huge_valf();
constexpr float LOG2E = 1.4426950408889634f;

// Error codes written to a translation unit's error word.
constexpr uint32_t ERR_WAIT_TIMEOUT = DFLASH2_DEVERR_WAIT_TIMEOUT;

// ------------------------------------------------------------------ PTX ----
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (TMA / tensor-core) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// One bounded poll of an mbarrier phase: the thread may be suspended for at
// most about 20 us while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// mbar_try_wait with a suspend-time hint of `ns` nanoseconds: the thread
// sleeps until the phase completes or about that long has passed.
__device__ __forceinline__ bool mbar_try_wait_ns(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// `max_cycles` SM clock cycles (the per-SM cycle counter is monotonic).
// Returns false on time-out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          long long max_cycles = 4000000000ll) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (clock64() - t0 <= max_cycles)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Order this thread's earlier generic-proxy accesses to shared memory before
// its later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// An L2 cache policy for data read once: its lines are evicted first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared (non-multicast), completing on `bar`, with
// an L2 cache policy for the lines it reads.  Both addresses 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s_hint(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_addr(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// Atomic add at GPU scope with acquire and release semantics: the writes
// that happen before it (this thread's, and those ordered before it by a
// __syncwarp) are visible to whoever acquires the result, and it sees the
// writes released by the atomics before it on the same word.
__device__ __forceinline__ int atomic_add_acq_rel(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Programmatic dependent launch.  pdl_wait: block until the grids this one
// depends on in the stream have completed and their memory is visible (a
// no-op when the grid was launched in the ordinary way).  pdl_trigger: let
// the next grid in the stream be launched before this one completes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Thread-block clusters.  cluster_sync: all threads of all CTAs of the
// cluster (release / acquire); the warp reconverges first.
__device__ __forceinline__ void cluster_sync() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store a 32-bit word into CTA `rank`'s shared memory at the address of
// `local` in this CTA (made visible to that CTA by the next cluster barrier).
__device__ __forceinline__ void st_dsmem_u32(void *local, uint32_t v, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// NaN-propagating maxima.
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 2^x on the special-function unit (relative error ~2^-22).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed f32x2 arithmetic (one instruction for two lanes of a 64-bit pair;
// low half first).  Each half is rounded as its scalar counterpart.
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint32_t lo32(uint64_t v) { return static_cast<uint32_t>(v); }
__device__ __forceinline__ uint32_t hi32(uint64_t v) { return static_cast<uint32_t>(v >> 32); }
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ------------------------------------------------------------ order keys ----
// A 64-bit key whose unsigned order is the candidate order: larger value
// first, then lower token id.  Key 0 is "empty" (below every real key).
__device__ __forceinline__ uint32_t f2ord(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord2f(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ uint64_t make_key(float v, uint32_t idx) {
    v = (v == 0.0f) ? 0.0f : v;  // -0 and +0 are one value: the id decides
    return (static_cast<uint64_t>(f2ord(v)) << 32) | static_cast<uint32_t>(~idx);
}
__device__ __forceinline__ float key_val(uint64_t k) { return ord2f(static_cast<uint32_t>(k >> 32)); }
__device__ __forceinline__ int32_t key_idx(uint64_t k) {
    return static_cast<int32_t>(~static_cast<uint32_t>(k));
}

// ----------------------------------------------------- warp top-N lists ----
// A warp holds R*32 keys sorted descending: position p = r*32 + lane.
template <int R>
struct WarpList {
    uint64_t k[R];
    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int r = 0; r < R; ++r) k[r] = 0;
    }
    // Key at position p (warp-uniform p).
    __device__ __forceinline__ uint64_t at(int p) const {
        uint64_t v = 0;
#pragma unroll
        for (int r = 0; r < R; ++r)
            if ((p >> 5) == r) v = __shfl_sync(FULL, k[r], p & 31);
        return v;
    }
    // Insert a warp-uniform key (distinct from every key present).
    __device__ __forceinline__ void insert(uint64_t key, int lane) {
        int pos = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) pos += __popc(__ballot_sync(FULL, k[r] > key));
        uint64_t carry = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            uint64_t up = __shfl_up_sync(FULL, k[r], 1);
            uint64_t last = __shfl_sync(FULL, k[r], 31);
            if (lane == 0) up = carry;
            carry = last;
            const int p = r * 32 + lane;
            k[r] = (p > pos) ? up : (p == pos ? key : k[r]);
        }
    }
    // this := top R*32 of (this U other), both sorted descending.
    __device__ __forceinline__ void merge(const WarpList &o, int lane) {
        // Reverse `o` and take the elementwise max: a bitonic sequence holding
        // the top R*32 of the union.
#pragma unroll
        for (int r = 0; r < R; ++r) {
            uint64_t rev = __shfl_sync(FULL, o.k[R - 1 - r], 31 - lane);
            k[r] = k[r] > rev ? k[r] : rev;
        }
        // Bitonic half-cleaners, descending.
        if (R == 2) {
            uint64_t a = k[0], b = k[R - 1];
            k[0] = a > b ? a : b;
            k[R - 1] = a > b ? b : a;
        }
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                uint64_t other = __shfl_xor_sync(FULL, k[r], d);
                const bool lower = (lane & d) == 0;
                k[r] = lower ? (k[r] > other ? k[r] : other) : (k[r] > other ? other : k[r]);
            }
        }
    }
    __device__ __forceinline__ void store(uint64_t *s, int lane) const {
#pragma unroll
        for (int r = 0; r < R; ++r) s[r * 32 + lane] = k[r];
    }
    __device__ __forceinline__ void load(const uint64_t *s, int lane) {
#pragma unroll
        for (int r = 0; r < R; ++r) k[r] = s[r * 32 + lane];
    }
};

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        uint64_t o = __shfl_xor_sync(FULL, v, d);
        v = v > o ? v : o;
    }
    return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, d));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(FULL, v, d);
    return v;
}

// Combine two (max, sum of 2^((x - max) * c)) pairs.
__device__ __forceinline__ void lse_combine(float &m, float &s, float m2, float s2, float c) {
    const float M = fmaxf(m, m2);
    if (M == NEG_INF) {
        m = M;
        s = 0.0f;
        return;
    }
    s = s * ex2((m - M) * c) + s2 * ex2((m2 - M) * c);
    m = M;
}

// --------------------------------------------------------- sampling rows ----
enum RowMode : int { MODE_ARGMAX = 0, MODE_TOPN_LSE = 1, MODE_TOPN = 2, MODE_SKIP = 3 };

struct RowTask {
    int mode;     // RowMode
    int nsel;     // list length the row needs
    int ek;       // effective top_k (V when off)
    int status;   // DFLASH2_ST_* reason for MODE_SKIP
    float T;      // temperature of the distribution (1 for greedy draft rows)
    float top_p;
    bool wide;    // a draft row whose filter may reach past its 64 best (top_k > 64, or top_p with top_k off)
};

// Decide how a row is scanned.  `target` rows need the target distribution
// p (argmax when greedy), draft rows the candidate list and U.
__device__ __forceinline__ RowTask decode_row(const dflash2_sampling *P, int64_t pidx, int64_t V,
                                              bool target) {
    RowTask t;
    t.wide = false;
    t.ek = static_cast<int>(V);
    t.status = DFLASH2_ST_OK;
    t.top_p = 1.0f;
    float T = 0.0f, tp = 1.0f;
    int tk = 0;
    if (P) {
        T = P[pidx].temperature;
        tk = P[pidx].top_k;
        tp = P[pidx].top_p;
    }
    if (!(T >= 0.0f) || isinf(T) || tk < 0 || !(tp > 0.0f && tp <= 1.0f)) {
        t.mode = MODE_SKIP;
        t.nsel = 0;
        t.T = 1.0f;
        t.status = DFLASH2_ST_BAD_PARAMS;
        return t;
    }
    if (T == 0.0f) {
        t.mode = target ? MODE_ARGMAX : MODE_TOPN_LSE;
        t.nsel = target ? 1 : NC;
        t.T = 1.0f;
        return t;
    }
    const int64_t ek = (tk == 0 || tk >= V) ? V : tk;
    const bool filtered = ek < V || tp < 1.0f;
    t.T = T;
    t.top_p = tp;
    if (!filtered) {
        t.mode = MODE_TOPN_LSE;
        if (target) {  // the whole row is p's support: the 64 best, the log normaliser, then passes
            t.nsel = DFLASH2_MAX_TOPK;
            t.ek = static_cast<int>(V);
            t.wide = true;
        } else {
            t.nsel = NC;
        }
        return t;
    }
    if (ek > DFLASH2_MAX_TOPK) {
        // the 64 best and the log normaliser; the cut may need passes over the row
        t.mode = MODE_TOPN_LSE;
        t.nsel = DFLASH2_MAX_TOPK;
        t.ek = static_cast<int>(ek);
        t.wide = true;
        return t;
    }
    t.ek = static_cast<int>(ek);
    t.mode = MODE_TOPN;
    t.nsel = target ? t.ek : (t.ek > NC ? t.ek : NC);
    return t;
}

}  // namespace dfl
