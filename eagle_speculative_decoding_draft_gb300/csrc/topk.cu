// topk.cu - per-row log-softmax and top-k over the vocabulary.
//
// EAGLE notes ch. 04 §10.2-§10.3: the confidence of a drafted token is its draft probability
// and every expanded node keeps its k most probable children.  Order: value descending, column
// ascending.  With k = 1 and no lse this is the target argmax of greedy verification.
//
// One thread-block cluster of C CTAs (C <= 8) per row; CTA r owns the r-th slice of the row and
// reads it from memory once, into registers:
//   pass 1  every thread takes the max of its elements.  The slice max and the slice threshold
//           (the largest, over warps, of the warp's k-th largest thread max: that warp alone has
//           k elements >= it) are pushed into every cluster CTA's shared memory; after a cluster
//           barrier every CTA takes the row max M and the row threshold tau as the max over the
//           cluster from its own copy (no remote loads).  Every element of the row's top k is
//           >= tau.
//   pass 2  from the registers: sum of exp2((x - M) log2 e) for the logsumexp, and every
//           element >= tau is appended to a shared candidate list; each candidate's rank in
//           the slice is the number of candidates that rank before it (one thread a candidate,
//           no sort), and the first k land in rank order.
//   merge   every CTA pushes its best k and its sum into rank 0's shared memory; after a second
//           cluster barrier rank 0 ranks the C x k entries the same way and writes the row's
//           top k and logsumexp.
// C shrinks when there are many rows, so that the grid fits in about one wave.
// k = 1 without the logsumexp (greedy verification's arg-max) takes a short path: the slices' best
// entries go to rank 0 and one cluster barrier separates them from the result.
// A slice with more than kCand elements >= tau (massive ties) falls back to k exact block-wide
// arg-max passes over that slice.
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
constexpr int kMaxCluster = 8;
constexpr int kCacheVec = 4;  // 16-byte vectors per thread held in registers between the passes
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// This CTA's part of the row: 16-byte vectors [vbeg, vend) and scalar elements [sbeg, send).
struct Slice {
    int32_t vbeg, vend, sbeg, send;
};

// Calls f(x, column) for every element of the slice: the first kCacheVec vectors of each thread
// come from `cache`, the rest (very long rows) and the scalar part from memory.
template <typename T, typename F>
__device__ __forceinline__ void visit(const T *z, const uint4 (&cache)[kCacheVec], const Slice &s,
                                      int32_t tid, F &&f) {
    constexpr int EPV = 16 / sizeof(T);
#pragma unroll
    for (int u = 0; u < kCacheVec; ++u) {
        const int32_t c = s.vbeg + tid + u * kThreads;
        if (c < s.vend) {
            const T *e = reinterpret_cast<const T *>(&cache[u]);
#pragma unroll
            for (int j = 0; j < EPV; ++j) f(to_f32(e[j]), c * EPV + j);
        }
    }
    // long rows: four vectors a thread and step, all loaded before any is used (same order of f)
    int32_t c = s.vbeg + kCacheVec * kThreads + tid;
    for (; c + 3 * kThreads < s.vend; c += 4 * kThreads) {
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
    for (; c < s.vend; c += kThreads) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(z) + c);
        const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
        for (int j = 0; j < EPV; ++j) f(to_f32(e[j]), c * EPV + j);
    }
    for (int32_t i = s.sbeg + tid; i < s.send; i += kThreads) f(to_f32(z[i]), i);
}

// Two CTAs per SM (64 registers a thread), so the CTAs of the next launch fit beside a GEMM CTA.
template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
    row_topk_kernel(const T *__restrict__ logits, int32_t V, int64_t ld, int32_t k,
                    int32_t *__restrict__ ids, float *__restrict__ vals, float *__restrict__ lse_out) {
    constexpr int EPV = 16 / sizeof(T);
    __shared__ float s_max[kWarps], s_kth[kWarps], s_sum[kWarps];
    __shared__ float c_v[kCand];
    __shared__ int32_t c_i[kCand];
    __shared__ int32_t s_count;
    __shared__ float r_v[kWarps];
    __shared__ int32_t r_i[kWarps];
    __shared__ float s_row[2];  // row max and threshold over the cluster
    __shared__ float p_stat[kMaxCluster][2];  // every slice's max and threshold, pushed by its CTA
    __shared__ float x_sum;      // this slice's sum of exp relative to the row max
    __shared__ float x_v[16];    // this slice's best k, sorted
    __shared__ int32_t x_i[16];
    // rank 0's inbox: every slice's sorted best k and its sum of exp
    __shared__ float m_v[kMaxCluster][16];
    __shared__ int32_t m_i[kMaxCluster][16];
    __shared__ float m_sum[kMaxCluster];
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const uint32_t C = cluster_size(), rank = cluster_rank();
    const int32_t row = blockIdx.x / C, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *z = logits + static_cast<int64_t>(row) * ld;
    const bool want_lse = lse_out != nullptr;

    // ---- this CTA's slice, loaded once ----
    const bool vec = (reinterpret_cast<uintptr_t>(z) % 16) == 0;
    const int32_t nvec = vec ? V / EPV : 0;
    const int32_t per = (nvec + static_cast<int32_t>(C) - 1) / static_cast<int32_t>(C);
    const int32_t rem = V - nvec * EPV;
    const int32_t sper = (rem + static_cast<int32_t>(C) - 1) / static_cast<int32_t>(C);
    Slice sl;
    sl.vbeg = min(nvec, static_cast<int32_t>(rank) * per);
    sl.vend = min(nvec, sl.vbeg + per);
    sl.sbeg = nvec * EPV + min(rem, static_cast<int32_t>(rank) * sper);
    sl.send = nvec * EPV + min(rem, static_cast<int32_t>(rank) * sper + sper);
    uint4 cache[kCacheVec];
#pragma unroll
    for (int u = 0; u < kCacheVec; ++u) {
        const int32_t c = sl.vbeg + tid + u * kThreads;
        cache[u] = (c < sl.vend) ? __ldg(reinterpret_cast<const uint4 *>(z) + c) : make_uint4(0, 0, 0, 0);
    }

    if (k == 1 && !want_lse) {
        // Arg-max only (greedy verification): the slice's best (value desc, id asc) by thread, warp
        // and block, pushed into rank 0, which takes the best of the C after one cluster barrier.
        float bv = -INFINITY;
        int32_t bi = INT_MAX;
        visit(z, cache, sl, tid, [&](float x, int32_t id) {
            if (before_nb(x, id, bv, bi)) {
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
        if (warp == 0) {
            float v = (lane < kWarps) ? r_v[lane] : -INFINITY;
            int32_t i = (lane < kWarps) ? r_i[lane] : INT_MAX;
            warp_best(v, i);
            if (lane == 0) {
                st_peer_f32(peer_addr(&m_v[rank][0], 0), v);
                st_peer_s32(peer_addr(&m_i[rank][0], 0), i);
            }
        }
        cluster_sync();
        if (rank == 0 && warp == 0) {
            float v = (lane < static_cast<int>(C)) ? m_v[lane][0] : -INFINITY;
            int32_t i = (lane < static_cast<int>(C)) ? m_i[lane][0] : INT_MAX;
            warp_best(v, i);
            if (lane == 0) {
                ids[row] = i;
                if (vals) vals[row] = v;
            }
        }
        return;
    }

    // ---- pass 1: thread max; slice max and threshold; row max and threshold ----
    float tmax = -INFINITY;
    visit(z, cache, sl, tid, [&](float x, int32_t) { tmax = fmaxf(tmax, x); });
    const float sorted = warp_sort_values(tmax, lane);
    const float wmax = __shfl_sync(kFullMask, sorted, 0);
    const float wkth = __shfl_sync(kFullMask, sorted, k - 1);
    if (lane == 0) {
        s_max[warp] = wmax;
        s_kth[warp] = wkth;
    }
    if (tid == 0) s_count = 0;
    __syncthreads();
    if (warp == 0) {
        float m = -INFINITY, t = -INFINITY;
        for (int w = 0; w < kWarps; ++w) {
            m = fmaxf(m, s_max[w]);
            t = fmaxf(t, s_kth[w]);
        }
        if (lane < static_cast<int>(C)) {  // push this slice's stats into CTA `lane`'s copy
            st_peer_f32(peer_addr(&p_stat[rank][0], lane), m);
            st_peer_f32(peer_addr(&p_stat[rank][1], lane), t);
        }
    }
    cluster_sync();  // every CTA's stats are in every CTA's p_stat
    if (warp == 0) {
        float m = -INFINITY, t = -INFINITY;
        if (lane < static_cast<int>(C)) {
            m = p_stat[lane][0];
            t = p_stat[lane][1];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
            t = fmaxf(t, __shfl_xor_sync(kFullMask, t, off));
        }
        if (lane == 0) {
            s_row[0] = m;
            s_row[1] = t;
        }
    }
    __syncthreads();
    const float M = s_row[0], tau = s_row[1];

    // ---- pass 2: sum of exp, candidates >= tau ----
    float sum = 0.0f;
    const float Ms = (M == -INFINITY) ? 0.0f : M * kLog2e;
    visit(z, cache, sl, tid, [&](float x, int32_t id) {
        if (want_lse) sum += exp2f(fmaf(x, kLog2e, -Ms));
        if (x >= tau) {
            const int32_t pos = atomicAdd(&s_count, 1);
            if (pos < kCand) {
                c_v[pos] = x;
                c_i[pos] = id;
            }
        }
    });
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFullMask, sum, off);
    if (lane == 0) s_sum[warp] = sum;
    __syncthreads();
    const int32_t count = s_count;
    if (tid == 0) {
        float tot = 0.0f;
        for (int w = 0; w < kWarps; ++w) tot += s_sum[w];
        x_sum = tot;
    }

    // ---- this slice's best k ----
    if (count <= kCand) {
        // rank of each candidate among the slice's candidates (a strict total order); the first
        // k go to their rank's slot, unfilled slots keep the (-inf, INT_MAX) sentinel
        if (tid < 16) {
            x_v[tid] = -INFINITY;
            x_i[tid] = INT_MAX;
        }
        __syncthreads();
        if (tid < count) {
            const float v = c_v[tid];
            const int32_t i = c_i[tid];
            int32_t r = 0;
            for (int32_t j = 0; j < count; ++j) r += before_nb(c_v[j], c_i[j], v, i) ? 1 : 0;
            if (r < k) {
                x_v[r] = v;
                x_i[r] = i;
            }
        }
    } else {
        // massive ties at the threshold: k exact passes, each the best element after the last pick
        float pv = INFINITY;
        int32_t pi = -1;
        for (int32_t j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int32_t bi = INT_MAX;
            visit(z, cache, sl, tid, [&](float x, int32_t id) {
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
                x_v[j] = bv;
                x_i[j] = bi;
            }
            pv = bv;
            pi = bi;
        }
    }
    __syncthreads();
    // ---- every slice's list and sum go to rank 0's inbox ----
    if (warp == 0) {
        if (lane < 16) {
            st_peer_f32(peer_addr(&m_v[rank][lane], 0), x_v[lane]);
            st_peer_s32(peer_addr(&m_i[rank][lane], 0), x_i[lane]);
        }
        if (lane == 0) st_peer_f32(peer_addr(&m_sum[rank], 0), x_sum);
    }
    // After this barrier no CTA touches a peer's shared memory again: rank 0 merges from its own.
    cluster_sync();

    // ---- rank 0 ranks the C x k entries of the slices' lists and writes the row's best k ----
    if (rank == 0) {
        if (warp == 0) {
            float tot = (lane < static_cast<int>(C)) ? m_sum[lane] : 0.0f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(kFullMask, tot, off);
            if (lane == 0) s_sum[0] = want_lse ? M + logf(tot) : 0.0f;
        }
        __syncthreads();
        const float lse = s_sum[0];
        const int32_t n = static_cast<int32_t>(C) * k;
        if (tid < n) {
            const int32_t p = tid / k, e = tid - p * k;
            const float v = m_v[p][e];
            const int32_t i = m_i[p][e];
            int32_t r = 0;
            for (int32_t q = 0; q < static_cast<int32_t>(C); ++q)
                for (int32_t f = 0; f < k; ++f) r += before_nb(m_v[q][f], m_i[q][f], v, i) ? 1 : 0;
            if (r < k) {  // sentinels rank after the >= k real entries of the row
                ids[static_cast<int64_t>(row) * k + r] = i;
                if (vals) vals[static_cast<int64_t>(row) * k + r] = want_lse ? v - lse : v;
            }
        }
        if (want_lse && tid == 0) lse_out[row] = lse;
    }
}

// Streaming multiprocessors of the current device (looked up once per device).
int sms_of_current_device() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

template <typename T>
cudaError_t launch_typed(const T *logits, int32_t rows, int32_t V, int64_t ld, int32_t k, int32_t *ids,
                         float *vals, float *lse, cudaStream_t st) {
    constexpr int EPV = 16 / sizeof(T);
    // about two vectors per thread per CTA, at most kMaxCluster CTAs, and no more CTAs than two
    // per SM in all (a power of two)
    const int64_t vecs = (static_cast<int64_t>(V) + EPV - 1) / EPV;
    int64_t c = (vecs + 2 * kThreads - 1) / (2 * kThreads);
    const int64_t fit = (2 * static_cast<int64_t>(sms_of_current_device())) / rows;
    if (c > fit) c = fit;
    if (c > kMaxCluster) c = kMaxCluster;
    unsigned C = 1;
    while (static_cast<int64_t>(C) * 2 <= c) C *= 2;
    return launch_pdl_cluster(row_topk_kernel<T>, dim3(static_cast<unsigned>(rows) * C), dim3(kThreads), C, 0,
                              st, logits, V, ld, k, ids, vals, lse);
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
