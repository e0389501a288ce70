// select.cuh - warp-level selection helpers: logsumexp merges, the warp's sorted values (a
// bitonic network on values only) and the warp's best (value, index).  Order everywhere: value
// descending, index ascending.
#pragma once

#include <climits>

#include "common.cuh"

namespace eagle {

constexpr unsigned kFullMask = 0xffffffffu;

__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
    const float nm = fmaxf(m, m2);
    if (nm == -INFINITY) {
        m = nm;
        s = 0.0f;
        return;
    }
    const float a = (m == -INFINITY) ? 0.0f : s * expf(m - nm);
    const float b = (m2 == -INFINITY) ? 0.0f : s2 * expf(m2 - nm);
    m = nm;
    s = a + b;
}

__device__ __forceinline__ void warp_lse(float &m, float &s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(kFullMask, m, off);
        const float s2 = __shfl_xor_sync(kFullMask, s, off);
        lse_merge(m, s, m2, s2);
    }
}

// Branch-free (a, ia) ranks strictly before (b, ib).
__device__ __forceinline__ bool before_nb(float a, int32_t ia, float b, int32_t ib) {
    return (a > b) | ((a == b) & (ia < ib));
}

// Values only: the warp's 32 values sorted descending across lanes (branch-free).
__device__ __forceinline__ float warp_sort_values(float v, int lane) {
#pragma unroll
    for (int k2 = 2; k2 <= 32; k2 <<= 1) {
#pragma unroll
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            const float o = __shfl_xor_sync(kFullMask, v, j);
            const bool keep_better = ((lane & j) == 0) == ((lane & k2) == 0);
            v = keep_better ? fmaxf(v, o) : fminf(v, o);
        }
    }
    return v;
}

// Warp-wide best of one (value, index) per lane; every lane gets the result.
__device__ __forceinline__ void warp_best(float &v, int32_t &i) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(kFullMask, v, off);
        const int32_t oi = __shfl_xor_sync(kFullMask, i, off);
        const bool take = before_nb(ov, oi, v, i);
        v = take ? ov : v;
        i = take ? oi : i;
    }
}

}  // namespace eagle
