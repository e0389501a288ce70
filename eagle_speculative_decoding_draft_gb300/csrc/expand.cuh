// expand.cuh - the expand step of one request, shared by expand_kernel and by the cluster row
// top-k kernel, whose last finishing row of a request runs it in the same launch.
//
// EAGLE notes ch. 04 §10.3 (expand: of the k^2 children of the newest level, keep the k with the
// highest scores S(child) = S(parent) + logp(child)); zdszero "在 SGLang 里" (top-k of k^2 per
// level).  Candidates are numbered level-major; every ranking is by (S descending, candidate
// ascending).
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace eagle {

struct ExpandSmem {
    float sS[256];
    int32_t sTok[256], sRow[256], sC[256];
    int32_t slot[16];
};

// Request b's candidates of this level (row_ids / row_logp of its rows, read through L2 when
// `from_l2`: they were written by other CTAs of the same launch), their pool entries and the
// next frontier (when `write_pool`).  All threads of the block call it (at least 256); returns
// false on the last level (no frontier), after which smem.slot is not valid.
__device__ __forceinline__ bool expand_request(const ExpandArgs &a, int32_t b, int32_t t, ExpandSmem &sm,
                                               bool write_pool, bool from_l2) {
    const int32_t k = a.k, kk = a.k * a.k;
    const int32_t nl = (a.level == 0) ? k : kk;
    if (t < nl) {
        int32_t tok, row, par, c;
        float S;
        if (a.level == 0) {
            row = b;
            const int64_t at = static_cast<int64_t>(b) * k + t;
            tok = from_l2 ? __ldcg(a.row_ids + at) : a.row_ids[at];
            S = from_l2 ? __ldcg(a.row_logp + at) : a.row_logp[at];
            par = -1;
            c = t;
        } else {
            const int32_t s = t / k, j = t - (t / k) * k;
            row = b * k + s;
            const int64_t at = static_cast<int64_t>(row) * k + j;
            tok = from_l2 ? __ldcg(a.row_ids + at) : a.row_ids[at];
            S = a.front_S_in[b * k + s] + (from_l2 ? __ldcg(a.row_logp + at) : a.row_logp[at]);
            par = a.front_cand_in[b * k + s];
            c = k + (a.level - 1) * kk + t;
            // the frontier holds candidates of the previous level
            if (!dcheck(par >= (a.level == 1 ? 0 : k + (a.level - 2) * kk) && par < k + (a.level - 1) * kk, a.status))
                par = 0;
        }
        if (!dcheck(c < a.n_cand, a.status)) c = 0;
        if (tok < 0 || tok >= a.V) {
            latch(a.status, kDevBounds);
            tok = 0;
        }
        sm.sS[t] = S;
        sm.sTok[t] = tok;
        sm.sRow[t] = row;
        sm.sC[t] = c;
        if (write_pool) {
            const int64_t o = static_cast<int64_t>(b) * a.n_cand + c;
            a.pool_tok[o] = tok;
            a.pool_S[o] = S;
            a.pool_parent[o] = par;
            a.pool_row[o] = row;
        }
    }
    if (a.front_cand_out == nullptr) return false;  // last level: no next frontier
    if (t < 16) sm.slot[t] = 0;  // every slot is overwritten when the scores are finite
    __syncthreads();
    if (t < nl) {
        int32_t rank = 0;
        for (int32_t u = 0; u < nl; ++u) rank += ranks_before(sm.sS[u], sm.sC[u], sm.sS[t], sm.sC[t]) ? 1 : 0;
        if (rank < k) sm.slot[rank] = t;
    }
    __syncthreads();
    if (t < k && !dcheck(sm.slot[t] >= 0 && sm.slot[t] < nl, a.status)) sm.slot[t] = 0;  // every rank < k is taken
    __syncthreads();
    if (write_pool && t < k) {
        a.front_cand_out[b * k + t] = sm.sC[sm.slot[t]];
        a.front_S_out[b * k + t] = sm.sS[sm.slot[t]];
    }
    return true;
}

}  // namespace eagle
