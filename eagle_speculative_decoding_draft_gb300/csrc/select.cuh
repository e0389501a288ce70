// select.cuh - warp-level selection by bitonic networks.  Order everywhere: value descending,
// index ascending.
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

// One compare-exchange step of a bitonic network across the warp.  keep_better: this lane keeps
// the better of the pair (else the worse).
// Branch-free (a, ia) ranks strictly before (b, ib).
__device__ __forceinline__ bool before_nb(float a, int32_t ia, float b, int32_t ib) {
    return (a > b) | ((a == b) & (ia < ib));
}

__device__ __forceinline__ void bitonic_step(float &v, int32_t &i, int j, bool keep_better) {
    const float ov = __shfl_xor_sync(kFullMask, v, j);
    const int32_t oi = __shfl_xor_sync(kFullMask, i, j);
    const bool ob = before_nb(ov, oi, v, i);
    const bool sb = before_nb(v, i, ov, oi);
    const bool take = (keep_better & ob) | ((!keep_better) & sb);
    v = take ? ov : v;
    i = take ? oi : i;
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

// Sorts the warp's 32 (value, index) pairs: lane 0 ends with the best.
__device__ __forceinline__ void warp_sort(float &v, int32_t &i, int lane) {
#pragma unroll
    for (int k2 = 2; k2 <= 32; k2 <<= 1) {
#pragma unroll
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            const bool lower = (lane & j) == 0;
            const bool desc = (lane & k2) == 0;
            bitonic_step(v, i, j, lower == desc);
        }
    }
}

// (v, i) is sorted across the warp; (bv, bi) is another sorted list.  Leaves in (v, i) the best
// 32 of both, sorted.
__device__ __forceinline__ void warp_merge_sorted(float &v, int32_t &i, float bv, int32_t bi, int lane) {
    const float rv = __shfl_sync(kFullMask, bv, 31 - lane);
    const int32_t ri = __shfl_sync(kFullMask, bi, 31 - lane);
    const bool take = before_nb(rv, ri, v, i);
    v = take ? rv : v;
    i = take ? ri : i;
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) bitonic_step(v, i, j, (lane & j) == 0);
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
