// sample.cu - sampling tree verification: recursive rejection sampling over the draft tree and
// its threshold variant.
//
// EAGLE notes ch. 04 §6.2: the target scores every tree node in one forward; then, from the root,
// a drafted token t is accepted when a uniform r satisfies r <= min(1, p(t) / q(t)); on rejection
// the distribution to draw from becomes norm(max(0, p - q)), and the next child is tested on it
// (SpecInfer's multi-candidate form, which the notes name as the framework).  When no child of
// the current node is accepted, the bonus token is drawn from the current distribution.  The
// threshold variant (the SGLang note in the summary of the tom-jerr EAGLE reading) accepts the
// first child whose target probability reaches a threshold and draws the bonus after one
// rejection step per child only when every child fails.
//
// Conventions: p = softmax(T[node] / temperature), q = softmax(Z[node] / temperature) (target
// and draft logits of the node, i.e. the distributions of the token after it); children are
// tested in ascending tree index with their own uniform u_acc[b][c]: accept iff p(t) > 0 and
// u * q(t) <= p(t); an empty residual leaves p unchanged; the bonus is the smallest token whose
// running sum of p (ascending ids) exceeds u_bonus * sum(p), else the largest token with p > 0.
//
// One thread-block cluster of C CTAs (C <= 8) per request; CTA r owns the r-th slice of the
// vocabulary.  The current distribution is kept implicit (computed from the target row) until
// the first rejection, then as an unnormalised row in the caller's scratch [B][V] times a scale.
// Every reduction is a block reduction followed by an exchange of the C partial results through
// distributed shared memory, summed in rank order, so every CTA of the cluster holds the same
// values and takes the same decisions: control flow stays uniform across the cluster.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.cuh"
#include "select.cuh"

namespace eagle {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;

struct SampleArgs {
    int32_t B, n, V, depth, mode;
    float inv_temp, threshold;
    const int32_t *tok, *par;
    const float *T, *Z, *u_acc, *u_bonus;
    float *scratch;
    int32_t *accept_len, *accept_nodes, *accept_tok;
};

__device__ __forceinline__ void online(float &m, float &s, float x) {
    if (x == -INFINITY) return;
    if (x > m) {
        s = (m == -INFINITY) ? 1.0f : s * __expf(m - x) + 1.0f;
        m = x;
    } else {
        s += __expf(x - m);
    }
}

// Cluster-wide reductions.  Each CTA pushes its values into slot `ph` of every cluster CTA's
// inbox before the barrier, and after it reads all of them from its own shared memory (no remote
// loads); `ph` flips, so a slot is written again only after every CTA has passed the barrier of
// the exchange that follows its last read of it.
struct Cluster {
    uint32_t C, rank;
    int ph;
    float *red;                      // kWarps floats (block partials)
    float (*inbox)[kMaxCluster][4];  // [2][C][4]: the values of every cluster CTA, by rank
    float *bc;                       // 4 floats: broadcast of the cluster result inside the CTA

    // Publishes up to 4 block-level values, then every thread returns the cluster result:
    // kind 0: sum of v[0]; kind 1: lse merge of (v[0], v[1]) and of (v[2], v[3]);
    // kind 2: (sum v0 in rank order, exclusive prefix of v0 before this rank, min v1, max v2).
    // v must hold the same values in every thread of the CTA.
    __device__ void exchange(const float (&v)[4], int kind, float (&out)[4]) {
        const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        if (tid < static_cast<int>(C)) {  // thread p pushes this CTA's values into CTA p's inbox
#pragma unroll
            for (int i = 0; i < 4; ++i) st_peer_f32(peer_addr(&inbox[ph][rank][i], tid), v[i]);
        }
        cluster_sync();
        if (warp == 0) {
            float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
            if (lane < static_cast<int>(C)) {
                a0 = inbox[ph][lane][0];
                a1 = inbox[ph][lane][1];
                a2 = inbox[ph][lane][2];
                a3 = inbox[ph][lane][3];
            }
            // combination over ranks 0..C-1 in a fixed order, identical on every CTA
            float o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f;
            if (kind == 1) {
                o0 = -INFINITY;
                o2 = -INFINITY;
            } else if (kind == 2) {
                o2 = __int_as_float(INT_MAX);
                o3 = __int_as_float(-1);
            }
            for (uint32_t r = 0; r < C; ++r) {
                const float b0 = __shfl_sync(kFullMask, a0, r), b1 = __shfl_sync(kFullMask, a1, r);
                const float b2 = __shfl_sync(kFullMask, a2, r), b3 = __shfl_sync(kFullMask, a3, r);
                if (kind == 0) {
                    o0 += b0;
                } else if (kind == 1) {
                    lse_merge(o0, o1, b0, b1);
                    lse_merge(o2, o3, b2, b3);
                } else {
                    if (r < rank) o1 += b0;
                    o0 += b0;
                    o2 = __int_as_float(min(__float_as_int(o2), __float_as_int(b1)));
                    o3 = __int_as_float(max(__float_as_int(o3), __float_as_int(b2)));
                }
            }
            if (lane == 0) {
                bc[0] = o0;
                bc[1] = o1;
                bc[2] = o2;
                bc[3] = o3;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) out[i] = bc[i];
        __syncthreads();  // bc is rewritten by the next exchange
        ph ^= 1;
    }
};

// Block-wide sum: every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.0f;
    for (int w = 0; w < kWarps; ++w) t += red[w];
    return t;
}

__global__ void __launch_bounds__(kThreads) verify_sample_kernel(const SampleArgs a) {
    __shared__ float red[kWarps], redm[kWarps], reds[kWarps];
    __shared__ int32_t redi[kWarps];
    __shared__ float inbox[2][kMaxCluster][4];
    __shared__ float bc[4];
    __shared__ int32_t kids[kMaxCandidates + 1];
    __shared__ int32_t s_nk;
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    Cluster cl{cluster_size(), cluster_rank(), 0, red, inbox, bc};
    const int32_t b = blockIdx.x / cl.C, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t n = a.n, V = a.V;
    // this CTA's slice of the vocabulary
    const int32_t per = (V + static_cast<int32_t>(cl.C) - 1) / static_cast<int32_t>(cl.C);
    const int32_t vb = min(V, static_cast<int32_t>(cl.rank) * per), ve = min(V, vb + per);
    const int32_t *tok = a.tok + static_cast<int64_t>(b) * n;
    const int32_t *par = a.par + static_cast<int64_t>(b) * n;
    float *scr = a.scratch + static_cast<int64_t>(b) * V;
    int32_t *an = a.accept_nodes + static_cast<int64_t>(b) * (a.depth + 1);
    int32_t *at = a.accept_tok + static_cast<int64_t>(b) * (a.depth + 1);
    const float it = a.inv_temp;

    int32_t cur = 0, nacc = 0;
    bool use_scr = false;
    float scale = 1.0f, lseT = 0.0f, lseZ = 0.0f;
    const float *trow = nullptr, *zrow = nullptr;
    // p(v) and q(v) of the current node, in the representation in force
    auto P = [&](int32_t v) -> float {
        return use_scr ? scr[v] * scale : __expf(fmaf(trow[v], it, -lseT));
    };
    auto Q = [&](int32_t v) -> float { return __expf(fmaf(zrow[v], it, -lseZ)); };
    float res[4];
    // P <- norm(max(0, P - q)); unchanged when the residual is empty
    auto residual = [&]() {
        float part = 0.0f;
        for (int32_t v = vb + tid; v < ve; v += kThreads) part += fmaxf(P(v) - Q(v), 0.0f);
        const float in[4] = {block_sum(part, red), 0.0f, 0.0f, 0.0f};
        cl.exchange(in, 0, res);
        const float S = res[0];
        if (S > 0.0f) {
            for (int32_t v = vb + tid; v < ve; v += kThreads) scr[v] = fmaxf(P(v) - Q(v), 0.0f);
            cluster_sync();  // the scratch row is read at any column by the next test
            use_scr = true;
            scale = 1.0f / S;
        }
    };

    for (;;) {
        trow = a.T + (static_cast<int64_t>(b) * n + cur) * V;
        zrow = a.Z + (static_cast<int64_t>(b) * n + cur) * V;
        use_scr = false;
        scale = 1.0f;
        // ---- logsumexp of T/temp and Z/temp in one pass over the slice ----
        float mt = -INFINITY, st = 0.0f, mz = -INFINITY, sz = 0.0f;
        for (int32_t v = vb + tid; v < ve; v += kThreads) {
            online(mt, st, trow[v] * it);
            online(mz, sz, zrow[v] * it);
        }
        warp_lse(mt, st);
        warp_lse(mz, sz);
        __syncthreads();
        if (lane == 0) {
            redm[warp] = mt;
            reds[warp] = st;
        }
        __syncthreads();
        float bm = -INFINITY, bs = 0.0f;
        for (int w = 0; w < kWarps; ++w) lse_merge(bm, bs, redm[w], reds[w]);
        __syncthreads();
        if (lane == 0) {
            redm[warp] = mz;
            reds[warp] = sz;
        }
        __syncthreads();
        float zm = -INFINITY, zs = 0.0f;
        for (int w = 0; w < kWarps; ++w) lse_merge(zm, zs, redm[w], reds[w]);
        const float in[4] = {bm, bs, zm, zs};
        cl.exchange(in, 1, res);
        lseT = res[0] + logf(res[1]);
        lseZ = res[2] + logf(res[3]);
        // ---- children of cur, in ascending index ----
        if (warp == 0) {
            int32_t cnt = 0;
            if (nacc < a.depth) {
                for (int32_t c0 = 1; c0 < n; c0 += 32) {
                    const int32_t c = c0 + lane;
                    const bool is = c < n && par[c] == cur;
                    const uint32_t m = __ballot_sync(kFullMask, is);
                    if (is) kids[cnt + __popc(m & ((1u << lane) - 1u))] = c;
                    cnt += __popc(m);
                }
            }
            if (lane == 0) s_nk = cnt;
        }
        __syncthreads();
        const int32_t nk = s_nk;
        int32_t next = -1;
        if (a.mode == 0) {
            for (int32_t j = 0; j < nk && next < 0; ++j) {
                const int32_t c = kids[j], t = tok[c];
                bool acc = false;
                if (t >= 0 && t < V) {
                    const float pt = P(t), qt = Q(t);
                    const float u = a.u_acc[static_cast<int64_t>(b) * n + c];
                    acc = pt > 0.0f && u * qt <= pt;
                }
                if (acc) next = c;
                else residual();
            }
        } else {
            for (int32_t j = 0; j < nk && next < 0; ++j) {
                const int32_t c = kids[j], t = tok[c];
                if (t >= 0 && t < V && P(t) >= a.threshold) next = c;
            }
            if (next < 0)
                for (int32_t j = 0; j < nk; ++j) residual();
        }
        __syncthreads();  // kids[] is rebuilt for the next node
        if (next < 0) break;
        if (cl.rank == 0 && tid == 0) {
            at[nacc] = tok[next];
            an[nacc + 1] = next;
        }
        ++nacc;
        cur = next;
    }

    // ---- bonus: inverse CDF of P over ascending ids ----
    // thread t of CTA r owns a contiguous chunk of the slice; chunk sums are scanned in thread
    // order, slice totals in rank order
    const int32_t len = ve - vb;
    const int32_t chunk = (len + kThreads - 1) / kThreads;
    const int32_t v0 = min(ve, vb + tid * chunk), v1 = min(ve, v0 + chunk);
    float csum = 0.0f;
    int32_t lastpos = -1;
    for (int32_t v = v0; v < v1; ++v) {
        const float pv = P(v);
        csum += pv;
        if (pv > 0.0f) lastpos = v;
    }
    float incl = csum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off) incl += o;
    }
    __syncthreads();
    if (lane == 31) reds[warp] = incl;
    __syncthreads();
    float wbase = 0.0f, slice = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) wbase += reds[w];
        slice += reds[w];
    }
    // slice totals over the cluster: the total and the exclusive prefix before this rank, both
    // summed in rank order
    {
        const float in[4] = {slice, __int_as_float(INT_MAX), __int_as_float(-1), 0.0f};
        cl.exchange(in, 2, res);
    }
    const float total = res[0], base = res[1];
    const float target = a.u_bonus[b] * total;
    float run = base + wbase + incl - csum;
    int32_t pick = INT_MAX;
    for (int32_t v = v0; v < v1; ++v) {
        const float pv = P(v);
        run += pv;
        if (run > target && pv > 0.0f) {
            pick = v;
            break;
        }
    }
    int32_t pm = pick, lm = lastpos;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        pm = min(pm, __shfl_xor_sync(kFullMask, pm, off));
        lm = max(lm, __shfl_xor_sync(kFullMask, lm, off));
    }
    __syncthreads();
    if (lane == 0) {
        redi[warp] = pm;
        redm[warp] = __int_as_float(lm);
    }
    __syncthreads();
    int32_t bp = INT_MAX, bl = -1;
    for (int w = 0; w < kWarps; ++w) {
        bp = min(bp, redi[w]);
        bl = max(bl, __float_as_int(redm[w]));
    }
    {
        const float in[4] = {0.0f, __int_as_float(bp), __int_as_float(bl), 0.0f};
        cl.exchange(in, 2, res);
    }
    if (cl.rank == 0 && tid == 0) {
        const int32_t best = __float_as_int(res[2]), last = __float_as_int(res[3]);
        at[nacc] = best != INT_MAX ? best : (last >= 0 ? last : 0);
        an[0] = 0;
        for (int32_t i = nacc + 1; i <= a.depth; ++i) {
            an[i] = -1;
            at[i] = -1;
        }
        a.accept_len[b] = nacc;
    }
    cluster_sync();  // peers' shared memory stays alive until every exchange has been read
}

}  // namespace

cudaError_t launch_verify_sample(int32_t B, int32_t n, int32_t V, int32_t depth, const int32_t *tok,
                                 const int32_t *par, const float *T, const float *Z, float temperature,
                                 int32_t mode, float threshold, const float *u_acc, const float *u_bonus,
                                 float *scratch, int32_t *accept_len, int32_t *accept_nodes,
                                 int32_t *accept_tok, cudaStream_t st) {
    if (B < 1) return cudaSuccess;
    SampleArgs a;
    a.B = B;
    a.n = n;
    a.V = V;
    a.depth = depth;
    a.mode = mode;
    a.inv_temp = 1.0f / temperature;
    a.threshold = threshold;
    a.tok = tok;
    a.par = par;
    a.T = T;
    a.Z = Z;
    a.u_acc = u_acc;
    a.u_bonus = u_bonus;
    a.scratch = scratch;
    a.accept_len = accept_len;
    a.accept_nodes = accept_nodes;
    a.accept_tok = accept_tok;
    // about 4096 vocabulary entries per CTA, at most kMaxCluster CTAs per request
    int32_t c = (V + 4095) / 4096;
    if (c < 1) c = 1;
    if (c > kMaxCluster) c = kMaxCluster;
    const unsigned C = static_cast<unsigned>(c);
    return launch_pdl_cluster(verify_sample_kernel, dim3(static_cast<unsigned>(B) * C), dim3(kThreads), C, 0, st,
                              a);
}

}  // namespace eagle
