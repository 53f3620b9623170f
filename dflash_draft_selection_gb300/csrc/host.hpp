// host.hpp -- host-side helpers of the DFlash 2 library: argument checks,
// device attributes and per-kernel occupancy, cached per device.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "dflash2.h"

namespace dfl {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

inline int sm_count() {
    static int cache[64] = {0};
    const int dev = current_device();
    if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

// Resident CTAs per SM of `func` with the given block and dynamic shared
// memory, after raising the kernel's dynamic shared-memory limit.  Cached per
// (kernel, device).
inline int blocks_per_sm(const void *func, int threads, size_t smem) {
    struct Entry {
        const void *f;
        int dev;
        int n;
    };
    static Entry cache[256];
    static int used = 0;
    static std::mutex mu;
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].f == func && cache[i].dev == dev) return cache[i].n;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem) != cudaSuccess || n < 1)
        n = 1;
    if (used < 256) cache[used++] = Entry{func, dev, n};
    return n;
}

// A launch attribute that lets this grid start while the previous grid in
// the stream is still running, as soon as that grid allows it (programmatic
// dependent launch); the grid itself waits (pdl_wait) before it reads what
// the previous grids wrote.
inline cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

inline dflash2_status after_launch() {
    return cudaPeekAtLastError() == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

inline int esize(dflash2_dtype dt) { return dt == DFLASH2_BF16 ? 2 : 4; }

inline bool dtype_ok(dflash2_dtype dt) { return dt == DFLASH2_BF16 || dt == DFLASH2_F32; }

// The merge of partials whose lists hold at most 16 entries (topk16.cu); the
// fused LM head's second launch.
dflash2_status launch_merge16(int S, int64_t rows, const int32_t *part_idx, const float *part_z, const float *part_m,
                              const float *part_s, int64_t V_total, const dflash2_sampling *params,
                              int64_t rows_per_param, int32_t *cand_idx, float *cand_U, float *lse,
                              cudaStream_t stream);

// gate = sigmoid(h . Wg^T) for checked arguments (gate.cu); the dynamic
// convolution's taps.  `early`: the grid may start beside the previous one.
dflash2_status gate_launch(const void *h, dflash2_dtype dt, int64_t n, int64_t hidden, const void *Wg, int D,
                           float *gate, cudaStream_t s, bool early);

}  // namespace dfl
