// topk.cu - per-row online log-softmax and top-k over the vocabulary.
//
// EAGLE notes ch. 04 §10.2-§10.3: the confidence of a drafted token is its draft probability
// and every expanded node keeps its k most probable children.  One CTA owns one row: its 512
// threads read the row with 16-byte loads, each keeping an online (max, sum of exp) pair and a
// sorted register list of its best KC elements; a warp merges its 32 lists by k rounds of
// shuffle-argmax (the winning lane pops its head), and warp 0 merges the 16 warp lists the same
// way.  Order: value descending, column ascending.  With k = 1 and no lse this is the target
// argmax of greedy verification.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.cuh"

namespace eagle {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <int KC>
struct TopList {
    float v[KC];
    int32_t i[KC];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int j = 0; j < KC; ++j) {
            v[j] = -INFINITY;
            i[j] = INT_MAX;
        }
    }
    __device__ __forceinline__ void insert(float x, int32_t id) {
        if (!ranks_before(x, id, v[KC - 1], i[KC - 1])) return;
        v[KC - 1] = x;
        i[KC - 1] = id;
#pragma unroll
        for (int j = KC - 1; j > 0; --j) {
            if (ranks_before(v[j], i[j], v[j - 1], i[j - 1])) {
                const float tv = v[j];
                v[j] = v[j - 1];
                v[j - 1] = tv;
                const int32_t ti = i[j];
                i[j] = i[j - 1];
                i[j - 1] = ti;
            }
        }
    }
    __device__ __forceinline__ void pop() {
#pragma unroll
        for (int j = 0; j < KC - 1; ++j) {
            v[j] = v[j + 1];
            i[j] = i[j + 1];
        }
        v[KC - 1] = -INFINITY;
        i[KC - 1] = INT_MAX;
    }
};

// Online softmax statistics: m = running max, s = sum of exp(x - m).
__device__ __forceinline__ void lse_add(float &m, float &s, float x) {
    if (!(x > -INFINITY)) return;  // -inf contributes nothing (NaN is ignored too)
    if (x > m) {
        s = s * expf(m - x) + 1.0f;
        m = x;
    } else {
        s += expf(x - m);
    }
}

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

// k rounds of warp-wide argmax over the lanes' list heads; the winning lane pops.  Every lane
// ends with the same `out` lists.
template <int KC>
__device__ __forceinline__ void warp_merge(TopList<KC> &list, int32_t k, float (&ov)[KC],
                                           int32_t (&oi)[KC]) {
#pragma unroll
    for (int j = 0; j < KC; ++j) {
        if (j < k) {
            float bv = list.v[0];
            int32_t bi = list.i[0];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float v2 = __shfl_xor_sync(0xffffffffu, bv, off);
                const int32_t i2 = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ranks_before(v2, i2, bv, bi)) {
                    bv = v2;
                    bi = i2;
                }
            }
            ov[j] = bv;
            oi[j] = bi;
            if (list.i[0] == bi && list.v[0] == bv) list.pop();
        } else {
            ov[j] = -INFINITY;
            oi[j] = INT_MAX;
        }
    }
}

template <int KC, typename T>
__global__ void __launch_bounds__(kThreads)
    row_topk_kernel(const T *__restrict__ logits, int32_t V, int64_t ld, int32_t k,
                    int32_t *__restrict__ ids, float *__restrict__ vals, float *__restrict__ lse_out) {
    __shared__ float s_v[kWarps][KC];
    __shared__ int32_t s_i[kWarps][KC];
    __shared__ float s_m[kWarps], s_s[kWarps];

    const int32_t row = blockIdx.x;
    const T *z = logits + static_cast<int64_t>(row) * ld;
    const bool want_lse = lse_out != nullptr;
    const int32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    TopList<KC> list;
    list.init();
    float m = -INFINITY, s = 0.0f;

    constexpr int EPV = 16 / sizeof(T);  // elements per 16-byte load
    const bool vec = (reinterpret_cast<uintptr_t>(z) % 16) == 0;
    const int32_t nvec = vec ? V / EPV : 0;
    for (int32_t c = tid; c < nvec; c += kThreads) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(z) + c);
        const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
            const float x = to_f32(e[j]);
            const int32_t id = c * EPV + j;
            if (want_lse) lse_add(m, s, x);
            list.insert(x, id);
        }
    }
    for (int32_t id = nvec * EPV + tid; id < V; id += kThreads) {
        const float x = to_f32(z[id]);
        if (want_lse) lse_add(m, s, x);
        list.insert(x, id);
    }

    float wv[KC];
    int32_t wi[KC];
    warp_merge<KC>(list, k, wv, wi);
    if (want_lse) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
            lse_merge(m, s, m2, s2);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < KC; ++j) {
            s_v[warp][j] = wv[j];
            s_i[warp][j] = wi[j];
        }
        s_m[warp] = m;
        s_s[warp] = s;
    }
    __syncthreads();
    if (warp != 0) return;

    list.init();
    if (lane < kWarps) {
#pragma unroll
        for (int j = 0; j < KC; ++j) {
            list.v[j] = s_v[lane][j];
            list.i[j] = s_i[lane][j];
        }
    }
    warp_merge<KC>(list, k, wv, wi);
    float lse = 0.0f;
    if (want_lse) {
        m = (lane < kWarps) ? s_m[lane] : -INFINITY;
        s = (lane < kWarps) ? s_s[lane] : 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
            lse_merge(m, s, m2, s2);
        }
        lse = m + logf(s);
    }
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < KC; ++j) {
            if (j < k) {
                ids[static_cast<int64_t>(row) * k + j] = wi[j];
                if (vals) vals[static_cast<int64_t>(row) * k + j] = want_lse ? wv[j] - lse : wv[j];
            }
        }
        if (want_lse) lse_out[row] = lse;
    }
}

template <typename T>
cudaError_t launch_typed(const T *logits, int32_t rows, int32_t V, int64_t ld, int32_t k, int32_t *ids,
                         float *vals, float *lse, cudaStream_t st) {
    const dim3 grid(rows), block(kThreads);
    if (k <= 1)
        row_topk_kernel<1, T><<<grid, block, 0, st>>>(logits, V, ld, k, ids, vals, lse);
    else if (k <= 2)
        row_topk_kernel<2, T><<<grid, block, 0, st>>>(logits, V, ld, k, ids, vals, lse);
    else if (k <= 4)
        row_topk_kernel<4, T><<<grid, block, 0, st>>>(logits, V, ld, k, ids, vals, lse);
    else if (k <= 8)
        row_topk_kernel<8, T><<<grid, block, 0, st>>>(logits, V, ld, k, ids, vals, lse);
    else
        row_topk_kernel<16, T><<<grid, block, 0, st>>>(logits, V, ld, k, ids, vals, lse);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_row_topk(const void *logits, int32_t is_bf16, int32_t rows, int32_t V, int64_t ld,
                            int32_t k, int32_t *ids, float *vals, float *lse, cudaStream_t st) {
    if (rows < 1) return cudaSuccess;
    if (is_bf16)
        return launch_typed(reinterpret_cast<const __nv_bfloat16 *>(logits), rows, V, ld, k, ids,
                            vals, lse, st);
    return launch_typed(reinterpret_cast<const float *>(logits), rows, V, ld, k, ids, vals, lse, st);
}

}  // namespace eagle
