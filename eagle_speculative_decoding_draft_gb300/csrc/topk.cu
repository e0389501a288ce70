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
#include "expand.cuh"
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
                    int32_t *__restrict__ ids, float *__restrict__ vals, float *__restrict__ lse_out,
                    const ExpandArgs ea, int32_t fx_rows, int32_t *fx_tickets) {
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
        if (fx_rows > 0) {
            // fused expand: the last of a request's rows to finish runs the request's expand
            __shared__ int32_t s_last;
            __shared__ ExpandSmem esm;
            __syncthreads();  // this row's ids and values are written
            const int32_t req = row / fx_rows;
            if (tid == 0) {
                __threadfence();  // release them before the ticket
                const int32_t prev = atomicAdd(&fx_tickets[req], 1);
                s_last = (prev == fx_rows - 1) ? 1 : 0;
                if (s_last) {
                    fx_tickets[req] = 0;  // ready for the next launch
                    __threadfence();      // and the other rows' results are read after this
                }
            }
            __syncthreads();
            if (s_last) expand_request(ea, req, tid, esm, true, true);
        }
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
                         float *vals, float *lse, cudaStream_t st, const FusedExpand *fx = nullptr) {
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
    ExpandArgs ea{};
    int32_t fx_rows = 0;
    int32_t *fx_tickets = nullptr;
    if (fx && fx->args) {
        ea = *fx->args;
        fx_rows = fx->rows_per_req;
        fx_tickets = fx->tickets;
    }
    return launch_pdl_cluster(row_topk_kernel<T>, dim3(static_cast<unsigned>(rows) * C), dim3(kThreads), C, 0,
                              st, logits, V, ld, k, ids, vals, lse, ea, fx_rows, fx_tickets);
}

// ---------------------------------------------------------------------------------------------
// Streaming row top-k for many long rows (rows at least the SM count, rows of at least 32 KB):
// one CTA a row reads it once, through a ring of 16 KB bulk copies (cp.async.bulk) into shared
// memory.  Warp 0 is the producer: it refills a stage as soon as the 16 consumer warps have
// released it (an mbarrier each way, no block-wide barrier in the loop), so the copies run ahead
// of the consumers by the whole ring.  Each consumer warp, with no barrier but its own:
//   lse     every thread sums exp(x - c) over its elements against its own offset c (its first
//           element, raised by rescaling only when an element exceeds it by more than 2^4); the
//           threads' (c, sum) pairs are merged by warps, then over the warps in a fixed order;
//   top k   the warp appends every element at or above its threshold to its own buffer (a
//           ballot a round, no atomics); when the buffer could overflow it keeps only its k best
//           (each entry ranked by counting, value descending, column ascending) and raises its
//           threshold to the k-th.  A row's top-k element is within its warp's k best,
//           so the warps' final k best, ranked the same way, give the row's top k exactly,
//           whatever the ties.
// k = 1 without the logsumexp (greedy verification's arg-max) keeps one best element a thread.
// ---------------------------------------------------------------------------------------------
constexpr int kStreamConsumers = 512;
constexpr int kStreamWarps = kStreamConsumers / 32;
constexpr int kStreamThreads = kStreamConsumers + 32;  // + the producer warp
constexpr uint32_t kChunkBytes = 16384;
constexpr int kStreamStages = 6;
constexpr int kWarpCap = 64;  // a warp's candidate buffer
constexpr int kSeedChunks = 4;  // chunks whose lane maxima give the first threshold
static_assert(kSeedChunks <= kStreamStages, "the seed's chunks are all in the ring at once");

struct StreamSmem {
    uint64_t full[kStreamStages];
    uint64_t empty[kStreamStages];
    float w_m[kStreamWarps], w_s[kStreamWarps], w_t[kStreamWarps];
    int32_t w_i[kStreamWarps];
    int32_t abort;
    float b_v[kStreamWarps][kWarpCap];  // the warps' candidates
    int32_t b_i[kStreamWarps][kWarpCap];
    float seed[kStreamWarps][16];  // each warp's k largest lane maxima of the first chunk
    float t0;                      // the k-th largest of them all: the warps' first threshold
};

// The consumers' common first threshold, from the first chunk: every lane's maximum over its
// elements there is one element of the row, so the k-th largest of the 512 lane maxima is at
// most the row's k-th largest value and no element of the row's top k falls below it.  Each
// warp sorts its 32 maxima and keeps its k largest; one warp then takes the k-th largest of
// those 16 sorted lists by k rounds that each remove the largest head.  Every consumer warp
// calls this once (two barriers over the 512 consumer threads).
__device__ __forceinline__ float stream_seed_threshold(StreamSmem *sm, float lane_max, int32_t warp, int32_t lane,
                                                       int32_t k) {
    const float sorted = warp_sort_values(lane_max, lane);
    if (lane < k) sm->seed[warp][lane] = sorted;
    named_barrier_sync(1, kStreamConsumers);
    if (warp == 0) {
        int32_t h = 0;  // this lane's list head (lanes below 16: warp `lane`'s list)
        float t = -INFINITY;
        for (int32_t r = 0; r < k; ++r) {
            const bool live = lane < kStreamWarps && h < k;
            const float v = live ? sm->seed[lane][h] : -INFINITY;
            float best = v;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) best = fmaxf(best, __shfl_xor_sync(kFullMask, best, off));
            const uint32_t hold = __ballot_sync(kFullMask, live && v == best);
            if (hold != 0u && lane == __ffs(hold) - 1) ++h;  // the lowest lane holding it moves on
            t = best;
        }
        if (lane == 0) sm->t0 = t;
    }
    named_barrier_sync(1, kStreamConsumers);
    return sm->t0;
}

// Keeps the k best of the warp's n <= 64 buffered entries (value descending, column ascending),
// in rank order at the front of the buffer; returns how many remain (min(n, k)) and sets thr to
// the k-th kept value when k are kept (-inf otherwise).  An element equal to it may still rank
// before it (a lower column appended later in the same round), so the filter is x >= thr and the
// next compaction settles the tie.
__device__ __forceinline__ int32_t warp_keep_best(float *bv, int32_t *bi, int32_t n, int32_t k, int32_t lane,
                                                  float &thr) {
    const float v0 = lane < n ? bv[lane] : -INFINITY, v1 = lane + 32 < n ? bv[lane + 32] : -INFINITY;
    const int32_t i0 = lane < n ? bi[lane] : INT_MAX, i1 = lane + 32 < n ? bi[lane + 32] : INT_MAX;
    int32_t r0 = 0, r1 = 0;
    for (int32_t j = 0; j < n; ++j) {
        const float u = bv[j];
        const int32_t ui = bi[j];
        r0 += ranks_before(u, ui, v0, i0) ? 1 : 0;
        r1 += ranks_before(u, ui, v1, i1) ? 1 : 0;
    }
    __syncwarp();
    if (lane < n && r0 < k) {
        bv[r0] = v0;
        bi[r0] = i0;
    }
    if (lane + 32 < n && r1 < k) {
        bv[r1] = v1;
        bi[r1] = i1;
    }
    __syncwarp();
    const int32_t kept = n < k ? n : k;
    thr = (kept == k) ? bv[k - 1] : -INFINITY;
    return kept;
}

template <typename T, bool kBestOnly>
__global__ void __launch_bounds__(kStreamThreads, 2)
    row_topk_stream_kernel(const T *__restrict__ logits, int32_t V, int64_t ld, int32_t k, int32_t *__restrict__ ids,
                           float *__restrict__ vals, float *__restrict__ lse_out, int32_t *status) {
    constexpr int EPV = 16 / sizeof(T);
    constexpr float kLog2e = 1.4426950408889634f;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw_addr + 127u) & ~127u) - raw_addr);
    StreamSmem *sm = reinterpret_cast<StreamSmem *>(ring + kStreamStages * kChunkBytes);
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    const int32_t row = blockIdx.x, lane = threadIdx.x & 31, warp = static_cast<int32_t>(threadIdx.x >> 5) - 1;
    const T *z = logits + static_cast<int64_t>(row) * ld;
    const uint32_t row_bytes = static_cast<uint32_t>(V) * sizeof(T);
    const int32_t nchunk = static_cast<int32_t>((row_bytes + kChunkBytes - 1) / kChunkBytes);
    const bool want_lse = lse_out != nullptr;
    if (threadIdx.x == 0) {
        for (int st = 0; st < kStreamStages; ++st) {
            mbar_init(&sm->full[st], 1);
            mbar_init(&sm->empty[st], kStreamWarps);
        }
        sm->abort = 0;
        sm->t0 = -INFINITY;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();  // the logits come from the previous kernel

    if (warp < 0) {
        // ---------------- producer: one thread refills each stage once the consumers release it ----
        if (lane == 0) {
            for (int32_t c = 0; c < nchunk; ++c) {
                const int st = c % kStreamStages;
                if (c >= kStreamStages &&
                    !mbar_wait(&sm->empty[st], static_cast<uint32_t>(c / kStreamStages - 1) & 1u, &sm->abort)) {
                    sm->abort = 1;
                    latch(status, kDevTimeout);
                    break;
                }
                const uint32_t off = static_cast<uint32_t>(c) * kChunkBytes;
                const uint32_t bytes = min(kChunkBytes, row_bytes - off);
                if (c >= kStreamStages) fence_proxy_async_smem();  // the consumers' reads, then the copy
                mbar_arrive_expect_tx(&sm->full[st], bytes);
                bulk_load(ring + st * kChunkBytes, reinterpret_cast<const uint8_t *>(z) + off, bytes, &sm->full[st]);
            }
        }
        __syncwarp();
    } else {
        // ---------------- 16 consumer warps ----------------
        float *wbv = sm->b_v[warp];
        int32_t *wbi = sm->b_i[warp];
        int32_t wn = 0;            // entries in this warp's buffer (the same in every lane)
        float thr = -INFINITY;     // this warp's threshold: an element below it cannot be in its k best
        float cof = -INFINITY, ssum = 0.0f;
        float bv = -INFINITY;  // arg-max only
        int32_t bi = INT_MAX;
        for (int32_t c = 0; c < nchunk; ++c) {
            const int st = c % kStreamStages;
            // one lane polls the stage's barrier while the others wait at the warp barrier (which
            // also orders the copy's bytes before their reads)
            int32_t got = 1;
            if (lane == 0) got = mbar_wait(&sm->full[st], static_cast<uint32_t>(c / kStreamStages) & 1u, &sm->abort);
            got = __shfl_sync(kFullMask, got, 0);
            __syncwarp();
            if (!got) {
                sm->abort = 1;
                latch(status, kDevTimeout);
            }
            const uint32_t bytes = min(kChunkBytes, row_bytes - static_cast<uint32_t>(c) * kChunkBytes);
            const int32_t nv = static_cast<int32_t>(bytes / 16u);
            const int32_t col0 = c * static_cast<int32_t>(kChunkBytes / sizeof(T));
            const uint8_t *stage = ring + st * kChunkBytes;
            if (!kBestOnly && c == 0) {
                // before any element is kept: a threshold from the lane maxima of the first
                // kSeedChunks chunks (already in the ring), so that few elements enter the
                // buffers and few rounds take the candidate path
                const int32_t nseed = min(nchunk, kSeedChunks);
                int32_t all = got;
                for (int32_t c2 = 1; c2 < nseed; ++c2) {
                    int32_t g2 = 1;
                    if (lane == 0) g2 = mbar_wait(&sm->full[c2], 0u, &sm->abort);
                    if (!__shfl_sync(kFullMask, g2, 0)) all = 0;
                }
                __syncwarp();
                if (!all) {
                    sm->abort = 1;
                    latch(status, kDevTimeout);
                }
                float lm = -INFINITY;  // fmaxf drops NaN: never NaN
                if (all)
                    for (int32_t c2 = 0; c2 < nseed; ++c2) {
                        const uint8_t *stg = ring + c2 * kChunkBytes;
                        const int32_t nv2 =
                            static_cast<int32_t>(min(kChunkBytes, row_bytes - static_cast<uint32_t>(c2) * kChunkBytes) / 16u);
                        for (int32_t v = warp * 32 + lane; v < nv2; v += kStreamConsumers) {
                            const uint4 raw = *reinterpret_cast<const uint4 *>(stg + v * 16);
                            const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
                            for (int j = 0; j < EPV; ++j) lm = fmaxf(lm, to_f32(e[j]));
                        }
                    }
                thr = stream_seed_threshold(sm, lm, warp, lane, k);
            }
            if (sm->abort) break;
            // two vectors a lane and round (v and v + 512 of the chunk: a thread still visits its
            // columns in ascending order); trips are warp-uniform
            for (int32_t va = warp * 32; va < nv; va += 2 * kStreamConsumers) {
                float x[2 * EPV];
                bool have[2];
                float cmax = -INFINITY;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int32_t v = va + u * kStreamConsumers + lane;
                    have[u] = v < nv;
                    if (have[u]) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(stage + v * 16);
                        const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
                        for (int j = 0; j < EPV; ++j) {
                            x[u * EPV + j] = to_f32(e[j]);
                            cmax = fmaxf(cmax, x[u * EPV + j]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < EPV; ++j) x[u * EPV + j] = -INFINITY;
                    }
                }
                if (kBestOnly) {
                    // an equal value later ranks after the thread's best
                    if (cmax > bv) {
#pragma unroll
                        for (int u = 0; u < 2; ++u)
#pragma unroll
                            for (int j = 0; j < EPV; ++j)
                                if (x[u * EPV + j] > bv) {
                                    bv = x[u * EPV + j];
                                    bi = col0 + (va + u * kStreamConsumers + lane) * EPV + j;
                                }
                    }
                    continue;
                }
                if (want_lse) {
                    if (cmax > cof + 16.0f) {  // keep the terms below 2^23: rescale to the new max
                        ssum = (cof == -INFINITY) ? 0.0f : ssum * ex2_approx((cof - cmax) * kLog2e);
                        cof = cmax;
                    }
                    if (cof != -INFINITY) {  // padding (-inf) adds exp(-inf) = 0
                        const float cl = cof * kLog2e;
                        float s0 = 0.0f, s1 = 0.0f;  // two chains of adds
#pragma unroll
                        for (int j = 0; j < 2 * EPV; j += 2) {
                            s0 += ex2_approx(fmaf(x[j], kLog2e, -cl));
                            s1 += ex2_approx(fmaf(x[j + 1], kLog2e, -cl));
                        }
                        ssum += s0 + s1;
                    }
                }
                if (__any_sync(kFullMask, cmax >= thr)) {
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int j = 0; j < EPV; ++j) {
                            bool in = have[u] && x[u * EPV + j] >= thr;
                            uint32_t ball = __ballot_sync(kFullMask, in);
                            if (ball == 0u) continue;
                            if (wn + __popc(ball) > kWarpCap) {
                                // full: keep the warp's k best, raise the threshold, vote again
                                wn = warp_keep_best(wbv, wbi, wn, k, lane, thr);
                                in = have[u] && x[u * EPV + j] >= thr;
                                ball = __ballot_sync(kFullMask, in);
                                if (ball == 0u) continue;
                            }
                            if (in) {
                                const int32_t pos = wn + __popc(ball & ((1u << lane) - 1u));
                                wbv[pos] = x[u * EPV + j];
                                wbi[pos] = col0 + (va + u * kStreamConsumers + lane) * EPV + j;
                            }
                            wn += __popc(ball);
                            __syncwarp();
                        }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm->empty[st]);  // this warp is done with the stage
        }
        if (!sm->abort) {
            if (kBestOnly) {
                warp_best(bv, bi);
                if (lane == 0) {
                    sm->w_t[warp] = bv;
                    sm->w_i[warp] = bi;
                }
            } else {
                wn = warp_keep_best(wbv, wbi, wn, k, lane, thr);
                if (lane == 0) sm->w_i[warp] = wn;
                float wm = cof, ws = ssum;
                warp_lse(wm, ws);
                if (lane == 0) {
                    sm->w_m[warp] = wm;
                    sm->w_s[warp] = ws;
                }
            }
        }
    }
    __syncthreads();  // also: every copy landed (the consumers waited on each) unless aborted
    if (sm->abort) {
        // let the copies in flight land before the CTA's shared memory is released
        if (threadIdx.x == 0) {
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < 200000ull) {
            }
        }
        __syncthreads();
        return;
    }
    const int32_t tid = static_cast<int32_t>(threadIdx.x);  // all 544 threads from here
    if (kBestOnly) {
        if (tid == 0) {
            float v = sm->w_t[0];
            int32_t i = sm->w_i[0];
            for (int w = 1; w < kStreamWarps; ++w)
                if (ranks_before(sm->w_t[w], sm->w_i[w], v, i)) {
                    v = sm->w_t[w];
                    i = sm->w_i[w];
                }
            ids[row] = i;
            if (vals) vals[row] = v;
        }
        return;
    }
    if (threadIdx.x >= 32) return;
    // one warp: the row's logsumexp (the warps' (max, sum) pairs merged in warp order), then the
    // k best of the warps' sorted lists by k rounds that each take the best head (value
    // descending, column ascending; a column is in one list only)
    float M = -INFINITY, S = 0.0f;
    if (want_lse) {
        if (lane == 0)
            for (int w = 0; w < kStreamWarps; ++w) lse_merge(M, S, sm->w_m[w], sm->w_s[w]);
        M = __shfl_sync(kFullMask, M, 0);
        S = __shfl_sync(kFullMask, S, 0);
    }
    const float lse = want_lse ? M + logf(S) : 0.0f;  // without it the values are the logits
    const int32_t n_l = lane < kStreamWarps ? sm->w_i[lane] : 0;
    int32_t h = 0;
    for (int32_t r = 0; r < k; ++r) {
        const bool live = h < n_l;
        float v = live ? sm->b_v[lane][h] : -INFINITY;
        int32_t c = live ? sm->b_i[lane][h] : INT_MAX;
        const int32_t mine = c;
        warp_best(v, c);
        if (c == INT_MAX) break;  // every list is empty
        if (live && mine == c) ++h;
        if (lane == 0) {
            ids[static_cast<int64_t>(row) * k + r] = c;
            if (vals) vals[static_cast<int64_t>(row) * k + r] = v - lse;
        }
    }
    if (lane == 0 && want_lse) lse_out[row] = lse;
}

constexpr size_t kStreamSmem = 128 + kStreamStages * kChunkBytes + sizeof(StreamSmem);

template <typename T>
cudaError_t launch_stream(const T *logits, int32_t rows, int32_t V, int64_t ld, int32_t k, int32_t *ids,
                          float *vals, float *lse, int32_t *status, cudaStream_t st) {
    static bool attr_set[64][4] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    auto go = [&](auto kernel, int slot) -> cudaError_t {
        if (dev >= 0 && dev < 64 && !attr_set[dev][slot]) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kStreamSmem));
            if (e != cudaSuccess) return e;
            attr_set[dev][slot] = true;
        }
        return launch_pdl(kernel, dim3(rows), dim3(kStreamThreads), kStreamSmem, st, logits, V, ld, k, ids, vals,
                          lse, status);
    };
    if (k == 1 && lse == nullptr) return go(row_topk_stream_kernel<T, true>, 0);
    return go(row_topk_stream_kernel<T, false>, 1);
}

// The streaming kernel serves many long rows whose starts and lengths suit 16-byte bulk copies:
// the arg-max from 32 KB rows on, the top k with the logsumexp from 2^16 elements on (below that
// the cluster kernel, which holds the row in registers, is faster: each warp's first candidates
// and the exp of every element cost more than its second read of a short row).
bool stream_suits(const void *logits, int32_t esize, int32_t rows, int32_t V, int64_t ld, bool best_only) {
    const int64_t bytes = static_cast<int64_t>(V) * esize;
    return rows >= sms_of_current_device() && bytes >= 32768 && (best_only || V >= 65536) && bytes % 16 == 0 &&
           (ld * esize) % 16 == 0 && (reinterpret_cast<uintptr_t>(logits) % 16) == 0;
}

}  // namespace

cudaError_t launch_row_topk(const void *logits, int32_t is_bf16, int32_t rows, int32_t V, int64_t ld,
                            int32_t k, int32_t *ids, float *vals, float *lse, cudaStream_t st, int32_t *status,
                            const FusedExpand *fx, bool *fused) {
    if (fused) *fused = false;
    if (rows < 1) return cudaSuccess;
    if (k >= 1 && k <= 16 && stream_suits(logits, is_bf16 ? 2 : 4, rows, V, ld, k == 1 && lse == nullptr)) {
        if (is_bf16)
            return launch_stream(reinterpret_cast<const __nv_bfloat16 *>(logits), rows, V, ld, k, ids, vals, lse,
                                 status, st);
        return launch_stream(reinterpret_cast<const float *>(logits), rows, V, ld, k, ids, vals, lse, status, st);
    }
    // the cluster kernel: it can run the level's expand (rows with logsumexp only)
    const bool fuse = fx && fx->args && lse != nullptr && fx->rows_per_req > 0 && fx->tickets != nullptr;
    if (fused) *fused = fuse;
    if (is_bf16)
        return launch_typed(reinterpret_cast<const __nv_bfloat16 *>(logits), rows, V, ld, k, ids, vals, lse, st,
                            fuse ? fx : nullptr);
    return launch_typed(reinterpret_cast<const float *>(logits), rows, V, ld, k, ids, vals, lse, st,
                        fuse ? fx : nullptr);
}

}  // namespace eagle
