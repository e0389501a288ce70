// topk.cu - per-row online log-softmax and top-k over the vocabulary.
//
// EAGLE notes ch. 04 §10.2-§10.3: the confidence of a drafted token is its draft probability
// and every expanded node keeps its k most probable children.  Order: value descending, column
// ascending.  With k = 1 and no lse this is the target argmax of greedy verification.
//
// Two kernels, so that a few rows still spread over the whole GPU:
//   partial  grid (rows, chunks): each 256-thread CTA reads one chunk of a row with 16-byte
//            loads issued up front, keeps an online (max, sum of exp) per lane, and a warp-wide
//            sorted list of the k best (lane j holds the j-th entry).  A batch of 32 elements
//            (one per lane) only touches the list when a ballot finds elements above the current
//            k-th; each such element is inserted with one ballot + one shuffle.  The 8 warp
//            lists are merged the same way and written with the chunk's (max, sum).
//   merge    one warp per row merges the chunks' lists and (max, sum) pairs, and writes the
//            ids, log-probabilities (value - lse) and lse.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.cuh"

namespace eagle {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

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

__device__ __forceinline__ void warp_lse(float &m, float &s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(kFull, m, off);
        const float s2 = __shfl_xor_sync(kFull, s, off);
        lse_merge(m, s, m2, s2);
    }
}

// A sorted list of the k best (value, index) pairs held across a warp: lane j < k holds entry j.
struct WarpList {
    float v;
    int32_t i;
    int32_t k;
    int32_t lane;
    __device__ __forceinline__ void init(int32_t k_, int32_t lane_) {
        v = -INFINITY;
        i = INT_MAX;
        k = k_;
        lane = lane_;
    }
    // The current k-th entry (the bar a candidate must clear).
    __device__ __forceinline__ void bar(float &bv, int32_t &bi) const {
        bv = __shfl_sync(kFull, v, k - 1);
        bi = __shfl_sync(kFull, i, k - 1);
    }
    // Inserts (cv, ci), known to rank before the k-th entry; warp-uniform arguments.
    __device__ __forceinline__ void insert(float cv, int32_t ci) {
        const uint32_t before = __ballot_sync(kFull, lane < k && ranks_before(v, i, cv, ci));
        const int32_t pos = __popc(before);
        const float uv = __shfl_up_sync(kFull, v, 1);
        const int32_t ui = __shfl_up_sync(kFull, i, 1);
        if (lane > pos) {
            v = uv;
            i = ui;
        } else if (lane == pos) {
            v = cv;
            i = ci;
        }
    }
    // Offers one candidate per lane; every candidate that belongs in the top k is inserted.
    __device__ __forceinline__ void offer(float x, int32_t id) {
        float bv;
        int32_t bi;
        bar(bv, bi);
        bool pending = ranks_before(x, id, bv, bi);
        uint32_t mask = __ballot_sync(kFull, pending);
        while (mask) {
            const int32_t src = __ffs(mask) - 1;
            const float cv = __shfl_sync(kFull, x, src);
            const int32_t ci = __shfl_sync(kFull, id, src);
            insert(cv, ci);
            bar(bv, bi);
            pending = pending && lane != src && ranks_before(x, id, bv, bi);
            mask = __ballot_sync(kFull, pending);
        }
    }
};

// Partial results of one (row, chunk): k values, k indices, max, sum.
struct Partials {
    float *val;      // [rows][chunks][k]
    int32_t *idx;    // [rows][chunks][k]
    float *m;        // [rows][chunks]
    float *s;        // [rows][chunks]
};

template <typename T, int EPT>
__global__ void __launch_bounds__(kThreads)
    topk_partial_kernel(const T *__restrict__ logits, int32_t V, int64_t ld, int32_t k,
                        int32_t want_lse, Partials p) {
    __shared__ float s_v[kWarps][32];
    __shared__ int32_t s_i[kWarps][32];
    __shared__ float s_m[kWarps], s_s[kWarps];
    const int32_t row = blockIdx.x, chunk = blockIdx.y, chunks = gridDim.y;
    const int32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *z = logits + static_cast<int64_t>(row) * ld;
    const int32_t base = chunk * kThreads * EPT;

    // ---- load this thread's EPT elements up front ----
    float x[EPT];
    int32_t id[EPT];
    constexpr int EPV = 16 / sizeof(T);
    const bool vec = (reinterpret_cast<uintptr_t>(z) % 16) == 0 && (EPT % EPV) == 0;
    if (vec) {
#pragma unroll
        for (int q = 0; q < EPT / EPV; ++q) {
            const int32_t e0 = base + (q * kThreads + tid) * EPV;
            if (e0 + EPV <= V) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(z + e0));
                const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
                for (int j = 0; j < EPV; ++j) {
                    x[q * EPV + j] = to_f32(e[j]);
                    id[q * EPV + j] = e0 + j;
                }
            } else {
#pragma unroll
                for (int j = 0; j < EPV; ++j) {
                    const int32_t e = e0 + j;
                    x[q * EPV + j] = (e < V) ? to_f32(z[e]) : -INFINITY;
                    id[q * EPV + j] = (e < V) ? e : INT_MAX;
                }
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const int32_t e = base + j * kThreads + tid;
            x[j] = (e < V) ? to_f32(z[e]) : -INFINITY;
            id[j] = (e < V) ? e : INT_MAX;
        }
    }

    // ---- per-lane softmax statistics, warp list ----
    float m = -INFINITY, s = 0.0f;
    if (want_lse) {
#pragma unroll
        for (int j = 0; j < EPT; ++j)
            if (id[j] != INT_MAX) lse_add(m, s, x[j]);
        warp_lse(m, s);
    }
    WarpList list;
    list.init(k, lane);
#pragma unroll
    for (int j = 0; j < EPT; ++j) list.offer(x[j], id[j]);

    // ---- merge the CTA's warp lists in warp 0 ----
    s_v[warp][lane] = list.v;
    s_i[warp][lane] = list.i;
    if (lane == 0) {
        s_m[warp] = m;
        s_s[warp] = s;
    }
    __syncthreads();
    if (warp != 0) return;
    for (int w = 1; w < kWarps; ++w) {
        const bool mine = lane < k;
        list.offer(mine ? s_v[w][lane] : -INFINITY, mine ? s_i[w][lane] : INT_MAX);
    }
    const int64_t slot = static_cast<int64_t>(row) * chunks + chunk;
    if (lane < k) {
        p.val[slot * k + lane] = list.v;
        p.idx[slot * k + lane] = list.i;
    }
    if (want_lse) {
        m = (lane < kWarps) ? s_m[lane] : -INFINITY;
        s = (lane < kWarps) ? s_s[lane] : 0.0f;
        warp_lse(m, s);
        if (lane == 0) {
            p.m[slot] = m;
            p.s[slot] = s;
        }
    }
}

// One warp per row: merge the row's chunk partials.
__global__ void __launch_bounds__(128)
    topk_merge_kernel(int32_t rows, int32_t chunks, int32_t k, int32_t want_lse, Partials p,
                      int32_t *__restrict__ ids, float *__restrict__ vals, float *__restrict__ lse_out) {
    const int32_t row = blockIdx.x * 4 + threadIdx.x / 32;
    const int32_t lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int64_t base = static_cast<int64_t>(row) * chunks;
    WarpList list;
    list.init(k, lane);
    const int32_t n = chunks * k;
    for (int32_t c0 = 0; c0 < n; c0 += 32) {
        const int32_t c = c0 + lane;
        const bool ok = c < n;
        list.offer(ok ? p.val[base * k + c] : -INFINITY, ok ? p.idx[base * k + c] : INT_MAX);
    }
    float lse = 0.0f;
    if (want_lse) {
        float m = -INFINITY, s = 0.0f;
        for (int32_t c = lane; c < chunks; c += 32) lse_merge(m, s, p.m[base + c], p.s[base + c]);
        warp_lse(m, s);
        lse = m + logf(s);
    }
    if (lane < k) {
        ids[static_cast<int64_t>(row) * k + lane] = list.i;
        if (vals) vals[static_cast<int64_t>(row) * k + lane] = want_lse ? list.v - lse : list.v;
    }
    if (want_lse && lane == 0) lse_out[row] = lse;
}

// Elements per thread of the partial kernel: enough CTAs to occupy the GPU, else bigger chunks.
int32_t choose_ept(int32_t rows, int32_t V) {
    const double elems = static_cast<double>(rows) * V;
    if (elems >= 600.0 * kThreads * 16) return 16;
    if (elems >= 300.0 * kThreads * 8) return 8;
    return 4;
}

Partials carve(void *ws, int32_t rows, int32_t chunks, int32_t k) {
    uint8_t *b = reinterpret_cast<uint8_t *>(ws);
    const size_t n = static_cast<size_t>(rows) * chunks;
    Partials p;
    p.val = reinterpret_cast<float *>(b);
    p.idx = reinterpret_cast<int32_t *>(b + n * k * 4);
    p.m = reinterpret_cast<float *>(b + 2 * n * k * 4);
    p.s = reinterpret_cast<float *>(b + 2 * n * k * 4 + n * 4);
    return p;
}

template <typename T>
cudaError_t launch_typed(const T *logits, int32_t rows, int32_t V, int64_t ld, int32_t k, int32_t *ids,
                         float *vals, float *lse, void *ws, cudaStream_t st) {
    const int32_t ept = choose_ept(rows, V);
    const int32_t chunks = (V + kThreads * ept - 1) / (kThreads * ept);
    const Partials p = carve(ws, rows, chunks, k);
    const int32_t want = lse != nullptr;
    const dim3 grid(rows, chunks);
    if (ept == 16)
        topk_partial_kernel<T, 16><<<grid, kThreads, 0, st>>>(logits, V, ld, k, want, p);
    else if (ept == 8)
        topk_partial_kernel<T, 8><<<grid, kThreads, 0, st>>>(logits, V, ld, k, want, p);
    else
        topk_partial_kernel<T, 4><<<grid, kThreads, 0, st>>>(logits, V, ld, k, want, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    topk_merge_kernel<<<(rows + 3) / 4, 128, 0, st>>>(rows, chunks, k, want, p, ids, vals, lse);
    return cudaGetLastError();
}

}  // namespace

size_t row_topk_scratch_bytes(int32_t rows, int32_t V, int32_t k) {
    // worst case is the smallest chunk (4 elements per thread)
    const size_t chunks = (static_cast<size_t>(V) + kThreads * 4 - 1) / (kThreads * 4);
    return static_cast<size_t>(rows) * chunks * (2 * static_cast<size_t>(k) + 2) * 4;
}

cudaError_t launch_row_topk(const void *logits, int32_t is_bf16, int32_t rows, int32_t V, int64_t ld,
                            int32_t k, int32_t *ids, float *vals, float *lse, void *ws, cudaStream_t st) {
    if (rows < 1) return cudaSuccess;
    if (is_bf16)
        return launch_typed(reinterpret_cast<const __nv_bfloat16 *>(logits), rows, V, ld, k, ids, vals,
                            lse, ws, st);
    return launch_typed(reinterpret_cast<const float *>(logits), rows, V, ld, k, ids, vals, lse, ws, st);
}

}  // namespace eagle
