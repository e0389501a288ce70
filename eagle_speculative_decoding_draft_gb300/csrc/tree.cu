// tree.cu - expand, rerank + tree build, greedy verify walk, and the row gather of the draft.
//
// EAGLE notes ch. 04 §10.3 (expand: keep the top-k nodes of the newest level; rerank: keep the
// top-m of all nodes; a child never outscores its parent so the kept set is a tree, ties to the
// shallower node), §12.5 (ancestor-only mask, positions shared per level), §6.2 (tree verify);
// zdszero "在 SGLang 里" (top-k of k^2 per level, top num_draft_tokens-1 overall, then the tree
// and mask); jsqmd "二、EAGLE-2" (flatten, positions, tree mask, longest consistent path).
//
// Scores are fp32 logs: S(child) = S(parent) + logp(child).  Every ranking is by
// (S descending, candidate ascending); candidates are numbered level-major, so a parent always
// ranks before its children and the kept set is closed under parents.
#include <climits>

#include <algorithm>

#include "common.cuh"
#include "expand.cuh"
#include "kernels.cuh"

namespace eagle {
namespace {

__device__ __forceinline__ int32_t cand_depth(int32_t c, int32_t k) {
    return c < k ? 1 : 2 + (c - k) / (k * k);
}

// ---------------------------------------------------------------------------------------------
// Expand.  Grid (B, Y): block (b, y) recomputes request b's candidates and their ranks (at most
// 256 of them); block y == 0 writes the pool and the next frontier; all Y blocks share the copy
// of the next level's rows [f^(producing row) || E[token]].
// ---------------------------------------------------------------------------------------------
constexpr int kExpandThreads = 256;

__global__ void __launch_bounds__(kExpandThreads) expand_kernel(const ExpandArgs a) {
    __shared__ ExpandSmem sm;
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t b = blockIdx.x, t = threadIdx.x, k = a.k;
    if (!expand_request(a, b, t, sm, blockIdx.y == 0, false)) return;
    const int32_t *slot = sm.slot, *sRow = sm.sRow, *sTok = sm.sTok;
    if (a.x_next == nullptr || a.fhat == nullptr) return;
    const int32_t eb = a.elem_bytes;
    const int32_t vpr = (2 * a.h * eb) / 16, vh = (a.h * eb) / 16;
    const uint8_t *fh = reinterpret_cast<const uint8_t *>(a.fhat);
    const uint8_t *em = reinterpret_cast<const uint8_t *>(a.emb);
    uint8_t *xo = reinterpret_cast<uint8_t *>(a.x_next);
    // two vectors a thread and step, both loads issued before either store
    const int32_t nv = k * vpr, stride = gridDim.y * kExpandThreads;
    for (int32_t i0 = blockIdx.y * kExpandThreads + t; i0 < nv; i0 += 2 * stride) {
        uint4 v[2];
        uint4 *to[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int32_t i = i0 + u * stride;
            to[u] = nullptr;
            if (i >= nv) continue;
            const int32_t sp = i / vpr, off = i - sp * vpr;
            const int32_t src = slot[sp];
            const uint4 *from = (off < vh)
                ? reinterpret_cast<const uint4 *>(fh + static_cast<int64_t>(sRow[src]) * a.h * eb) + off
                : reinterpret_cast<const uint4 *>(em + static_cast<int64_t>(sTok[src]) * a.h * eb) + (off - vh);
            to[u] = reinterpret_cast<uint4 *>(xo + static_cast<int64_t>(b * k + sp) * 2 * a.h * eb) + off;
            v[u] = __ldg(from);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
            if (to[u]) *to[u] = v[u];
    }
}

// ---------------------------------------------------------------------------------------------
// Rerank + build: one CTA per request.
// ---------------------------------------------------------------------------------------------
constexpr int kBuildThreads = 512;

// Order-preserving unsigned key of a float: a < b (as floats, no NaN) iff key(a) < key(b).
__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t u = (x == 0.0f) ? 0u : __float_as_uint(x);  // -0 and +0 compare equal
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide sum of one int per thread; `red` holds kBuildThreads / 32 ints.
__device__ __forceinline__ int32_t block_total(int32_t v, int32_t *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();  // `red` may still be read by the previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int32_t s = 0;
#pragma unroll
    for (int w = 0; w < kBuildThreads / 32; ++w) s += red[w];
    return s;
}

__global__ void __launch_bounds__(kBuildThreads) build_tree_kernel(const BuildArgs a) {
    extern __shared__ int32_t sm[];
    const int32_t nc = a.n_cand, n = a.m + 1;
    float *sS = reinterpret_cast<float *>(sm);
    int32_t *sPar = sm + nc;
    int32_t *sIdx = sPar + nc;  // tree index of a kept candidate, 0 if not kept
    int32_t *tPar = sIdx + nc;  // parent tree index of each node
    __shared__ int32_t warp_cnt[kBuildThreads / 32], warp_off[kBuildThreads / 32], running;
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();

    const int32_t b = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t pb = static_cast<int64_t>(b) * nc;
    for (int32_t c = t; c < nc; c += kBuildThreads) {
        sS[c] = a.pool_S[pb + c];
        sPar[c] = a.pool_parent[pb + c];
    }
    __syncthreads();
    // Kept iff fewer than m candidates rank before it by (S descending, id ascending).  Radix
    // select of the m-th largest score on order-preserving keys (32 block-wide counts), then the
    // candidates tied with it are kept in id order up to m.
    uint32_t thr = 0;  // key of the m-th largest score
    int32_t above = 0;  // candidates strictly above it
    if (a.m > 0 && nc <= kBuildThreads) {
        // one candidate per thread: each step is one counting barrier
        const uint32_t key = (t < nc) ? order_key(sS[t]) : 0u;
        const bool real = t < nc;
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = thr | (1u << bit);
            if (__syncthreads_count(real && key >= cand) >= a.m) thr = cand;
        }
        above = __syncthreads_count(real && key > thr);
    } else if (a.m > 0) {
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = thr | (1u << bit);
            int32_t cnt = 0;
            for (int32_t c = t; c < nc; c += kBuildThreads) cnt += (order_key(sS[c]) >= cand) ? 1 : 0;
            if (block_total(cnt, warp_cnt) >= a.m) thr = cand;
        }
        int32_t cnt = 0;
        for (int32_t c = t; c < nc; c += kBuildThreads) cnt += (order_key(sS[c]) > thr) ? 1 : 0;
        above = block_total(cnt, warp_cnt);
    }
    if (t == 0) running = 0;
    __syncthreads();
    // ties with the m-th score, in id order: the first m - above of them are kept
    for (int32_t base = 0; base < nc; base += kBuildThreads) {
        const int32_t c = base + t;
        const uint32_t key = (c < nc) ? order_key(sS[c]) : 0u;
        const bool tie = a.m > 0 && c < nc && key == thr;
        const uint32_t ballot = __ballot_sync(0xffffffffu, tie);
        if (lane == 0) warp_cnt[warp] = __popc(ballot);
        __syncthreads();
        if (t == 0) {
            int32_t acc = 0;
            for (int w = 0; w < kBuildThreads / 32; ++w) {
                warp_off[w] = acc;
                acc += warp_cnt[w];
            }
        }
        __syncthreads();
        if (c < nc) {
            const int32_t eq_rank = running + warp_off[warp] + __popc(ballot & ((1u << lane) - 1u));
            sIdx[c] = (a.m > 0 && (key > thr || (tie && eq_rank < a.m - above))) ? 1 : 0;
        }
        __syncthreads();
        if (t == 0) running += warp_off[kBuildThreads / 32 - 1] + warp_cnt[kBuildThreads / 32 - 1];
        __syncthreads();
    }
    if (t == 0) running = 0;
    __syncthreads();
    // tree index = 1 + number of kept candidates with a smaller id (block scan, chunk by chunk)
    for (int32_t base = 0; base < nc; base += kBuildThreads) {
        const int32_t c = base + t;
        const int32_t flag = (c < nc) ? sIdx[c] : 0;
        const uint32_t ballot = __ballot_sync(0xffffffffu, flag);
        if (lane == 0) warp_cnt[warp] = __popc(ballot);
        __syncthreads();
        if (t == 0) {
            int32_t acc = 0;
            for (int w = 0; w < kBuildThreads / 32; ++w) {
                warp_off[w] = acc;
                acc += warp_cnt[w];
            }
        }
        __syncthreads();
        if (flag) sIdx[c] = 1 + running + warp_off[warp] + __popc(ballot & ((1u << lane) - 1u));
        __syncthreads();
        if (t == 0) running += warp_off[kBuildThreads / 32 - 1] + warp_cnt[kBuildThreads / 32 - 1];
        __syncthreads();
    }
    const int64_t ob = static_cast<int64_t>(b) * n;
    const int32_t pos0 = a.pos_base ? a.pos_base[b] : 0;
    for (int32_t i = t; i < n; i += kBuildThreads) tPar[i] = (i == 0) ? -1 : 0;
    __syncthreads();
    if (t == 0) {
        a.tokens[ob] = a.root_tok[b];
        a.parents[ob] = -1;
        a.positions[ob] = pos0;
        if (a.logscore) a.logscore[ob] = 0.0f;
        if (a.node_tok) a.node_tok[ob] = a.root_tok[b];
        if (a.node_src) a.node_src[ob] = -1 - b;
    }
    for (int32_t c = t; c < nc; c += kBuildThreads) {
        const int32_t ti = sIdx[c];
        if (ti <= 0 || ti >= n) continue;
        const int32_t pc = sPar[c];
        int32_t pt = 0;
        if (pc >= nc) {
            latch(a.status, kDevBounds);
        } else if (pc >= 0) {
            pt = sIdx[pc];
            if (pt <= 0) {  // parent not kept: impossible for finite scores
                latch(a.status, kDevTree);
                pt = 0;
            }
        }
        tPar[ti] = pt;
        const int32_t dep = cand_depth(c, a.k);
        const int32_t tok = a.pool_tok[pb + c];
        a.tokens[ob + ti] = tok;
        a.parents[ob + ti] = pt;
        a.positions[ob + ti] = dep + pos0;
        if (a.logscore) a.logscore[ob + ti] = sS[c];
        if (a.node_tok) a.node_tok[ob + ti] = tok;
        if (a.node_src && a.pool_row) {
            int32_t prow = a.pool_row[pb + c];
            if (!dcheck(prow >= 0 && prow < a.r_pad && dep >= 1 && dep <= a.d, a.status)) prow = 0;
            a.node_src[ob + ti] = (dep - 1) * a.r_pad + prow;
        }
    }
    __syncthreads();
    // ancestor-only mask, LSB-first bits: walk up the parents (strictly decreasing indices)
    const int32_t W = (n + 31) / 32;
    for (int32_t ti = t; ti < n; ti += kBuildThreads) {
        for (int32_t w = 0; w < W; ++w) {
            uint32_t word = 0;
            for (int32_t x = ti; x >= 0; x = tPar[x])
                if ((x >> 5) == w) word |= 1u << (x & 31);
            a.mask[(ob + ti) * W + w] = word;
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Verify walk: one warp per request.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128)
    verify_walk_kernel(int32_t B, int32_t n, int32_t d, const int32_t *__restrict__ tok,
                       const int32_t *__restrict__ par, const int32_t *__restrict__ g,
                       int32_t *accept_len, int32_t *accept_nodes, int32_t *accept_tok) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t b = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int32_t lane = threadIdx.x & 31;
    if (b >= B) return;
    const int32_t *tk = tok + static_cast<int64_t>(b) * n;
    const int32_t *pr = par + static_cast<int64_t>(b) * n;
    const int32_t *gb = g + static_cast<int64_t>(b) * n;
    int32_t *an = accept_nodes + static_cast<int64_t>(b) * (d + 1);
    int32_t *at = accept_tok + static_cast<int64_t>(b) * (d + 1);
    for (int32_t i = lane; i <= d; i += 32) {
        an[i] = -1;
        at[i] = -1;
    }
    __syncwarp();
    int32_t cur = 0, L = 0, gc = gb[0];
    if (lane == 0) an[0] = 0;
    while (L < d) {
        int32_t next = INT_MAX;
        for (int32_t i = 1 + lane; i < n; i += 32)
            if (pr[i] == cur && tk[i] == gc) next = min(next, i);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) next = min(next, __shfl_xor_sync(0xffffffffu, next, off));
        if (next == INT_MAX) break;
        if (lane == 0) {
            at[L] = tk[next];
            an[L + 1] = next;
        }
        ++L;
        cur = next;
        gc = gb[cur];
    }
    if (lane == 0) {
        at[L] = gc;
        accept_len[b] = L;
    }
}

// ---------------------------------------------------------------------------------------------
// Row gather: X[r] = [feature || E[token]].
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gather_kernel(const GatherArgs a) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t r = blockIdx.x;
    int32_t si = a.src ? a.src[r] : -1 - r;
    // a source row: f^ row si of the handle's levels, or root feature -1 - si
    if (a.src_rows > 0 && !dcheck(si < a.src_rows && -1 - si < a.root_rows, a.status)) si = -1;
    int32_t tok = a.tok[r];
    if (a.tok_copy && blockIdx.y == 0 && threadIdx.x == 0) a.tok_copy[r] = tok;
    if (tok < 0 || tok >= a.V) {
        if (threadIdx.x == 0 && blockIdx.y == 0) latch(a.status, kDevBounds);
        tok = 0;
    }
    const int32_t eb = a.elem_bytes;
    const int32_t vpr = (2 * a.h * eb) / 16, vh = (a.h * eb) / 16;
    const uint8_t *fsrc = (si >= 0)
        ? reinterpret_cast<const uint8_t *>(a.fhat_all) + static_cast<int64_t>(si) * a.h * eb
        : reinterpret_cast<const uint8_t *>(a.root_feat) + static_cast<int64_t>(-1 - si) * a.h * eb;
    const uint8_t *esrc = reinterpret_cast<const uint8_t *>(a.emb) + static_cast<int64_t>(tok) * a.h * eb;
    uint4 *to = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(a.x) + static_cast<int64_t>(r) * 2 * a.h * eb);
    for (int32_t i = blockIdx.y * blockDim.x + threadIdx.x; i < vpr; i += gridDim.y * blockDim.x)
        to[i] = (i < vh) ? __ldg(reinterpret_cast<const uint4 *>(fsrc) + i)
                         : __ldg(reinterpret_cast<const uint4 *>(esrc) + (i - vh));
}

// ---------------------------------------------------------------------------------------------
// Draft extend (zdszero "在 SGLang 里"): row r = b (d+1) + i is [F[b][a_j] || E[t_j]] with
// j = min(i, L_b), a_j / t_j the accepted path's j-th node and the token that follows it
// (L_b = accept_len[b]).  The row of the last verified position also gives the next round's
// root: its feature and token, and the root token kept for the tree build.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) extend_gather_kernel(const ExtendArgs a) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t r = blockIdx.x, d1 = a.d + 1;
    const int32_t b = r / d1, i = r - b * d1;
    int32_t L = a.accept_len[b];
    if (L < 0 || L > a.d) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && i == 0) latch(a.status, kDevBounds);
        L = L < 0 ? 0 : a.d;
    }
    const int32_t j = i < L ? i : L;
    int32_t node = a.accept_nodes[static_cast<int64_t>(b) * d1 + j];
    int32_t tok = a.accept_tok[static_cast<int64_t>(b) * d1 + j];
    if (node < 0 || node >= a.n || tok < 0 || tok >= a.V) {
        if (threadIdx.x == 0 && blockIdx.y == 0) latch(a.status, kDevBounds);
        node = (node < 0 || node >= a.n) ? 0 : node;
        tok = (tok < 0 || tok >= a.V) ? 0 : tok;
    }
    const int32_t eb = a.elem_bytes;
    const int32_t vh = (a.h * eb) / 16, vpr = 2 * vh;
    const uint4 *fsrc = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(a.node_feat) +
                                                        (static_cast<int64_t>(b) * a.n + node) * a.h * eb);
    const uint4 *esrc = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(a.emb) +
                                                        static_cast<int64_t>(tok) * a.h * eb);
    uint4 *to = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(a.x) + static_cast<int64_t>(r) * 2 * a.h * eb);
    for (int32_t v = blockIdx.y * blockDim.x + threadIdx.x; v < vpr; v += gridDim.y * blockDim.x)
        to[v] = (v < vh) ? __ldg(fsrc + v) : __ldg(esrc + (v - vh));
    if (i == L) {
        uint4 *nf = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(a.next_feat) + static_cast<int64_t>(b) * a.h * eb);
        for (int32_t v = blockIdx.y * blockDim.x + threadIdx.x; v < vh; v += gridDim.y * blockDim.x) nf[v] = __ldg(fsrc + v);
        if (threadIdx.x == 0 && blockIdx.y == 0) {
            a.next_tok[b] = tok;
            a.root_tok[b] = tok;
        }
    }
}

// Level 0's f^ row of request b = the extend's row of its last verified position; optionally every
// path row to the caller.
__global__ void __launch_bounds__(256) extend_select_kernel(const ExtendArgs a) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t b = blockIdx.x, d1 = a.d + 1;
    int32_t L = a.accept_len[b];
    L = L < 0 ? 0 : (L > a.d ? a.d : L);
    const int32_t eb = a.elem_bytes, vh = (a.h * eb) / 16;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.ext_fhat);
    uint4 *lvl0 = reinterpret_cast<uint4 *>(a.fhat0);
    for (int32_t v = blockIdx.y * blockDim.x + threadIdx.x; v < vh; v += gridDim.y * blockDim.x)
        lvl0[static_cast<int64_t>(b) * vh + v] = src[(static_cast<int64_t>(b) * d1 + L) * vh + v];
    if (a.path_fhat) {
        uint4 *out = reinterpret_cast<uint4 *>(a.path_fhat);
        for (int32_t v = blockIdx.y * blockDim.x + threadIdx.x; v < d1 * vh; v += gridDim.y * blockDim.x)
            out[static_cast<int64_t>(b) * d1 * vh + v] = src[static_cast<int64_t>(b) * d1 * vh + v];
    }
}

// ---------------------------------------------------------------------------------------------
// EAGLE-1 static tree ("EAGLE notes ch. 04" §10.1, §12 item 7): block (b, c) handles node
// lo + c of depth level+1 for request b.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) static_expand_kernel(const StaticExpandArgs a) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t b = blockIdx.x, j = a.lo + blockIdx.y, n = a.n;
    const int32_t p = a.sp[kSpPar * n + j], r = a.sp[kSpRank * n + j];
    const int32_t row = b * a.E + a.sp[kSpPeidx * n + j];
    int32_t tok = a.row_ids[static_cast<int64_t>(row) * a.K + r];
    if (tok < 0 || tok >= a.V) {
        if (threadIdx.x == 0) latch(a.status, kDevBounds);
        tok = 0;
    }
    if (threadIdx.x == 0) {
        const float Sp = (a.level == 0) ? 0.0f : a.node_S[static_cast<int64_t>(b) * n + p];
        a.node_tok[static_cast<int64_t>(b) * n + j] = tok;
        a.node_S[static_cast<int64_t>(b) * n + j] = Sp + a.row_logp[static_cast<int64_t>(row) * a.K + r];
    }
    const int32_t e = a.sp[kSpEidx * n + j];
    if (a.x_next == nullptr || e < 0) return;
    const int32_t eb = a.elem_bytes, vh = (a.h * eb) / 16;
    const uint4 *f = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(a.fhat) +
                                                     static_cast<int64_t>(row) * a.h * eb);
    const uint4 *em = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(a.emb) +
                                                      static_cast<int64_t>(tok) * a.h * eb);
    uint4 *to = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(a.x_next) +
                                          static_cast<int64_t>(b * a.E_next + e) * 2 * a.h * eb);
    for (int32_t v = threadIdx.x; v < 2 * vh; v += blockDim.x) to[v] = (v < vh) ? __ldg(f + v) : __ldg(em + (v - vh));
}

__global__ void __launch_bounds__(256) static_build_kernel(const StaticBuildArgs a) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t b = blockIdx.x, n = a.n;
    const int64_t ob = static_cast<int64_t>(b) * n;
    const int32_t pos0 = a.pos_base ? a.pos_base[b] : 0;
    for (int32_t j = threadIdx.x; j < n; j += blockDim.x) {
        const int32_t tok = (j == 0) ? a.root_tok[b] : a.node_tok[ob + j];
        a.tokens[ob + j] = tok;
        a.parents[ob + j] = a.sp[kSpPar * n + j];
        a.positions[ob + j] = a.sp[kSpDep * n + j] + pos0;
        if (a.logscore) a.logscore[ob + j] = (j == 0) ? 0.0f : a.node_S[ob + j];
        for (int32_t w = 0; w < a.W; ++w) a.mask[(ob + j) * a.W + w] = a.sp_mask[static_cast<int64_t>(j) * a.W + w];
        if (j == 0) {
            a.node_tok[ob] = tok;
            a.node_src[ob] = -1 - b;
        } else {
            a.node_src[ob + j] = a.sp[kSpSrcOff * n + j] + b * a.sp[kSpEStride * n + j] + a.sp[kSpPeidx * n + j];
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Test hook: one thread waits, with the bounded wait every device wait of the library uses, on an
// mbarrier that nothing will ever arrive on; when the limit passes it latches the timeout bit in
// the status word and returns.  Proves the timeout path without faulting or hanging anything.
// ---------------------------------------------------------------------------------------------
__global__ void bounded_wait_kernel(uint64_t limit_ns, int32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait(&bar, 0, nullptr, limit_ns)) latch(status, kDevTimeout);
}

}  // namespace

cudaError_t launch_expand(const ExpandArgs &a, cudaStream_t st) {
    if (a.B < 1) return cudaSuccess;
    int32_t y = 1;
    if (a.x_next && a.fhat) {
        const int64_t bytes = static_cast<int64_t>(a.k) * 2 * a.h * a.elem_bytes;
        y = static_cast<int32_t>((bytes + 8191) / 8192);  // about 8 KB of copy per block
        if (y < 1) y = 1;
        if (y > 64) y = 64;
    }
    return launch_pdl(expand_kernel, dim3(a.B, y), dim3(kExpandThreads), 0, st, a);
}

cudaError_t launch_build_tree(const BuildArgs &a, cudaStream_t st) {
    if (a.B < 1) return cudaSuccess;
    const size_t smem = (3 * static_cast<size_t>(a.n_cand) + a.m + 1) * sizeof(int32_t);
    return launch_pdl(build_tree_kernel, dim3(a.B), dim3(kBuildThreads), smem, st, a);
}

cudaError_t prepare_tree_kernels() {
    return cudaFuncSetAttribute(build_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>((3 * kMaxCandidates + kMaxCandidates + 1) * 4));
}

cudaError_t launch_verify_walk(int32_t B, int32_t n, int32_t d, const int32_t *tok, const int32_t *par,
                               const int32_t *g, int32_t *accept_len, int32_t *accept_nodes,
                               int32_t *accept_tok, cudaStream_t st) {
    if (B < 1) return cudaSuccess;
    return launch_pdl(verify_walk_kernel, dim3((B + 3) / 4), dim3(128), 0, st, B, n, d, tok, par, g, accept_len,
                      accept_nodes, accept_tok);
}

cudaError_t launch_gather(const GatherArgs &a, cudaStream_t st) {
    if (a.n_rows < 1) return cudaSuccess;
    const int64_t bytes = 2LL * a.h * a.elem_bytes;
    int32_t y = static_cast<int32_t>((bytes + 4095) / 4096);
    if (y < 1) y = 1;
    return launch_pdl(gather_kernel, dim3(a.n_rows, y), dim3(256), 0, st, a);
}

cudaError_t launch_bounded_wait(uint64_t limit_ns, int32_t *status, cudaStream_t st) {
    bounded_wait_kernel<<<1, 32, 0, st>>>(limit_ns, status);
    return cudaGetLastError();
}

cudaError_t launch_extend_gather(const ExtendArgs &a, cudaStream_t st) {
    const int32_t rows = a.B * (a.d + 1);
    if (rows < 1) return cudaSuccess;
    const int32_t y = std::max(1, std::min(8, (2 * a.h * a.elem_bytes) / 4096));
    return launch_pdl(extend_gather_kernel, dim3(rows, y), dim3(256), 0, st, a);
}

cudaError_t launch_extend_select(const ExtendArgs &a, cudaStream_t st) {
    if (a.B < 1) return cudaSuccess;
    const int32_t y = std::max(1, std::min(8, (a.h * a.elem_bytes) / 4096));
    return launch_pdl(extend_select_kernel, dim3(a.B, y), dim3(256), 0, st, a);
}

cudaError_t launch_static_expand(const StaticExpandArgs &a, cudaStream_t st) {
    if (a.B < 1 || a.cnt < 1) return cudaSuccess;
    return launch_pdl(static_expand_kernel, dim3(a.B, a.cnt), dim3(128), 0, st, a);
}

cudaError_t launch_static_build(const StaticBuildArgs &a, cudaStream_t st) {
    if (a.B < 1) return cudaSuccess;
    return launch_pdl(static_build_kernel, dim3(a.B), dim3(256), 0, st, a);
}

}  // namespace eagle
