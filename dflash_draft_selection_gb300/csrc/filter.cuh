// filter.cuh -- the sampling filter on a row's best keys, shared by the draft
// (U of the filtered drafter distribution) and the target (p of the verify).
// FreeToken PR 857 "Speed": temperature 1.0, top_p 0.95, top_k 20 on both
// sides; filters applied as temperature -> top_k -> renormalise -> top_p ->
// renormalise.
#pragma once

#include "common.cuh"

namespace dfl {

__device__ __forceinline__ float warp_inclusive_scan(float v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float t = __shfl_up_sync(FULL, v, d);
        if (lane >= d) v += t;
    }
    return v;
}

// The sampling filter on a row's best keys (temperature -> top_k ->
// renormalise -> top_p -> renormalise).  Returns the kept count; e[r] holds
// exp((z_p - z_0) / T) for the position p = r*32 + lane (0 past top_k) and
// *ekept the sum over the kept positions.  Warp-uniform.
template <int R>
__device__ __forceinline__ int topn_filter(const WarpList<R> &L, const RowTask &task, float z0,
                                           int lane, float (&e)[R], float *ekept) {
    float part = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int p = r * 32 + lane;
        e[r] = (p < task.ek) ? expf((key_val(L.k[r]) - z0) / task.T) : 0.0f;
        part += e[r];
    }
    const float Ek = warp_sum(part);
    int kept = task.ek;
    if (task.top_p < 1.0f) {
        const float thr = task.top_p * Ek;
        float base = 0.0f;
        bool found = false;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float cum = warp_inclusive_scan(e[r], lane) + base;
            const int p = r * 32 + lane;
            const uint32_t hit = __ballot_sync(FULL, p < task.ek && cum >= thr);
            if (hit && !found) {
                kept = r * 32 + __ffs(hit);
                found = true;
            }
            base = __shfl_sync(FULL, cum, 31);
        }
    }
    float kp = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r)
        if (r * 32 + lane < kept) kp += e[r];
    *ekept = warp_sum(kp);
    return kept;
}

}  // namespace dfl
