// topk.cu - per-row log-softmax and top-k over the vocabulary.
//
// EAGLE notes ch. 04 §10.2-§10.3: the confidence of a drafted token is its draft probability
// and every expanded node keeps its k most probable children.  Order: value descending, column
// ascending.  With k = 1 and no lse this is the target argmax of greedy verification.
//
// One CTA per row, two passes over the row (the second one hits L2):
//   pass 1  every thread takes the max of its elements; the row max M is the block max, and the
//           threshold tau is the largest, over warps, of the warp's k-th largest thread max: that
//           warp alone has k elements >= tau, so every element of the top k is >= tau.
//   pass 2  sum of exp2((x - M) log2 e) for the logsumexp, and every element >= tau (usually a
//           few more than k) is appended to a shared candidate list.
//   select  one warp sorts the candidates with bitonic networks and keeps the first k.
// A row with more than kCand elements >= tau (massive ties) falls back to k exact block-wide
// arg-max passes.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.cuh"
#include "select.cuh"

namespace eagle {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCand = 256;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// Calls f(x, index) for every element of the row; 16-byte loads when the row is aligned.
template <typename T, typename F>
__device__ __forceinline__ void for_each(const T *z, int32_t V, int32_t tid, F &&f) {
    constexpr int EPV = 16 / sizeof(T);
    const bool vec = (reinterpret_cast<uintptr_t>(z) % 16) == 0;
    const int32_t nvec = vec ? V / EPV : 0;
    int32_t c = tid;
    for (; c + 3 * kThreads < nvec; c += 4 * kThreads) {
        uint4 raw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) raw[u] = __ldg(reinterpret_cast<const uint4 *>(z) + c + u * kThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const T *e = reinterpret_cast<const T *>(&raw[u]);
#pragma unroll
            for (int j = 0; j < EPV; ++j) f(to_f32(e[j]), (c + u * kThreads) * EPV + j);
        }
    }
    for (; c < nvec; c += kThreads) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(z) + c);
        const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
        for (int j = 0; j < EPV; ++j) f(to_f32(e[j]), c * EPV + j);
    }
    for (int32_t id = nvec * EPV + tid; id < V; id += kThreads) f(to_f32(z[id]), id);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    row_topk_kernel(const T *__restrict__ logits, int32_t V, int64_t ld, int32_t k,
                    int32_t *__restrict__ ids, float *__restrict__ vals, float *__restrict__ lse_out) {
    __shared__ float s_max[kWarps], s_kth[kWarps], s_sum[kWarps];
    __shared__ float c_v[kCand];
    __shared__ int32_t c_i[kCand];
    __shared__ int32_t s_count;
    __shared__ float r_v[kWarps];
    __shared__ int32_t r_i[kWarps];
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *z = logits + static_cast<int64_t>(row) * ld;
    const bool want_lse = lse_out != nullptr;

    // ---- pass 1: thread max, row max, threshold ----
    float tmax = -INFINITY;
    for_each(z, V, tid, [&](float x, int32_t) { tmax = fmaxf(tmax, x); });
    const float sorted = warp_sort_values(tmax, lane);
    const float wmax = __shfl_sync(kFullMask, sorted, 0);
    const float wkth = __shfl_sync(kFullMask, sorted, k - 1);
    if (lane == 0) {
        s_max[warp] = wmax;
        s_kth[warp] = wkth;
    }
    if (tid == 0) s_count = 0;
    __syncthreads();
    float M = -INFINITY, tau = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        M = fmaxf(M, s_max[w]);
        tau = fmaxf(tau, s_kth[w]);
    }

    // ---- pass 2: sum of exp, candidates >= tau ----
    float sum = 0.0f;
    const float Ms = (M == -INFINITY) ? 0.0f : M * kLog2e;
    for_each(z, V, tid, [&](float x, int32_t id) {
        if (want_lse) sum += exp2f(fmaf(x, kLog2e, -Ms));
        if (x >= tau) {
            const int32_t pos = atomicAdd(&s_count, 1);
            if (pos < kCand) {
                c_v[pos] = x;
                c_i[pos] = id;
            }
        }
    });
    if (want_lse) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFullMask, sum, off);
        if (lane == 0) s_sum[warp] = sum;
    }
    __syncthreads();
    const int32_t count = s_count;
    float lse = 0.0f;
    if (want_lse) {
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tot += s_sum[w];
        lse = M + logf(tot);
    }

    // ---- select the top k ----
    if (count <= kCand) {
        if (warp == 0) {
            float v = -INFINITY;
            int32_t i = INT_MAX;
            for (int32_t b0 = 0; b0 < count; b0 += 32) {
                float bv = (b0 + lane < count) ? c_v[b0 + lane] : -INFINITY;
                int32_t bi = (b0 + lane < count) ? c_i[b0 + lane] : INT_MAX;
                warp_sort(bv, bi, lane);
                if (b0 == 0) {
                    v = bv;
                    i = bi;
                } else {
                    warp_merge_sorted(v, i, bv, bi, lane);
                }
            }
            if (lane < k) {
                ids[static_cast<int64_t>(row) * k + lane] = i;
                if (vals) vals[static_cast<int64_t>(row) * k + lane] = want_lse ? v - lse : v;
            }
            if (want_lse && lane == 0) lse_out[row] = lse;
        }
        return;
    }
    // massive ties at the threshold: k exact passes, each the best element after the previous pick
    float pv = INFINITY;
    int32_t pi = -1;
    for (int32_t j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int32_t bi = INT_MAX;
        for_each(z, V, tid, [&](float x, int32_t id) {
            const bool after = before_nb(pv, pi, x, id);  // ranks after the previous pick
            if (after && before_nb(x, id, bv, bi)) {
                bv = x;
                bi = id;
            }
        });
        warp_best(bv, bi);
        if (lane == 0) {
            r_v[warp] = bv;
            r_i[warp] = bi;
        }
        __syncthreads();
        bv = r_v[0];
        bi = r_i[0];
        for (int w = 1; w < kWarps; ++w)
            if (before_nb(r_v[w], r_i[w], bv, bi)) {
                bv = r_v[w];
                bi = r_i[w];
            }
        __syncthreads();
        if (tid == 0) {
            ids[static_cast<int64_t>(row) * k + j] = bi;
            if (vals) vals[static_cast<int64_t>(row) * k + j] = want_lse ? bv - lse : bv;
        }
        pv = bv;
        pi = bi;
    }
    if (want_lse && tid == 0) lse_out[row] = lse;
}

template <typename T>
cudaError_t launch_typed(const T *logits, int32_t rows, int32_t V, int64_t ld, int32_t k, int32_t *ids,
                         float *vals, float *lse, cudaStream_t st) {
    return launch_pdl(row_topk_kernel<T>, dim3(rows), dim3(kThreads), 0, st, logits, V, ld, k, ids, vals, lse);
}

}  // namespace

cudaError_t launch_row_topk(const void *logits, int32_t is_bf16, int32_t rows, int32_t V, int64_t ld,
                            int32_t k, int32_t *ids, float *vals, float *lse, cudaStream_t st) {
    if (rows < 1) return cudaSuccess;
    if (is_bf16)
        return launch_typed(reinterpret_cast<const __nv_bfloat16 *>(logits), rows, V, ld, k, ids, vals, lse, st);
    return launch_typed(reinterpret_cast<const float *>(logits), rows, V, ld, k, ids, vals, lse, st);
}

}  // namespace eagle
