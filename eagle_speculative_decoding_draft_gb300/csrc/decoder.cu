// decoder.cu - the draft decoder layer: one Llama decoder layer over the nodes of each request's
// draft tree, with tree attention over a draft KV cache.
//
// zdszero, "在 SGLang 里": the draft model is the embedding, fc = Linear(2h, h, bias), one Llama
// decoder layer whose first input_layernorm is the identity, no final norm, and the target's
// lm_head.  EAGLE notes ch. 04 §4.1 (FC, then a light decoder layer predicts the next feature) and
// §12.5 (tree attention: a node sees its ancestors only).  Per node i of request b:
//   qkv = Wqkv x_i; q, k rotated (Llama rotate-half RoPE) at pos[b][i]
//   o   = softmax over the P cached keys and the tree keys that node i's mask row marks
//   h1  = x_i + Wo o;  r = RMSNorm(h1) * w_norm;  a = silu(g) * u with [g; u] = Wgu r
//   out = h1 + Wd a
// Each projection output, the attention output, each residual sum, r and a are rounded to bf16;
// dot products, softmax and norms are fp32.  The four projections run on the streamed-weight
// tcgen05 GEMM (gemm.cu); this file holds the attention and the element-wise kernels.
#include <algorithm>
#include <cfloat>
#include <mutex>

#include "../../include/eagle_tree.h"
#include "common.cuh"
#include "kernels.cuh"
#include "select.cuh"

namespace eagle {
namespace {

__device__ __forceinline__ float bf(const __nv_bfloat16 v) { return __bfloat162float(v); }

constexpr int kMaxHeadDim = 128;

// RoPE in place on the q and k parts of each qkv row: pair (j, j + D/2) of every head rotated by
// pos * theta^(-2j/D).  Block (row, head slice).  The frequency theta^(-2j/D) is base^j with
// base = theta^(-2/D) (one pow per block, then binary powering: a dozen double roundings at most),
// computed before the wait on the previous kernel; the angle pos * freq is formed and reduced
// mod 2 pi in double, and only the reduced angle (|r| <= pi) goes to fp32 sincosf: the cosine and
// sine carry ~1e-7 absolute error, against the 2^-9 relative half-ulp of the bf16 outputs.  One
// (cos, sin) per pair serves all heads of the row.  Each thread turns 4 consecutive pairs of a head.
// With k_new / v_new the rotated keys and the values of the row are also written there.
__global__ void __launch_bounds__(256) rope_kernel(__nv_bfloat16 *qkv, int32_t nqkv, int32_t H, int32_t Hk,
                                                   int32_t heads_per_block, int32_t D, const int32_t *pos,
                                                   double theta, __nv_bfloat16 *k_new, __nv_bfloat16 *v_new) {
    __shared__ double s_base;
    __shared__ float2 s_cs[kMaxHeadDim / 2];
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    const int32_t half = D / 2, row = blockIdx.x;
    if (threadIdx.x == 0) s_base = pow(theta, -2.0 / static_cast<double>(D));
    __syncthreads();
    double f = 1.0;
    if (threadIdx.x < half) {
        double b = s_base;
        for (int32_t e = threadIdx.x; e; e >>= 1) {
            if (e & 1) f *= b;
            b *= b;
        }
    }
    pdl_wait();  // positions and qkv may come from earlier kernels
    if (threadIdx.x < half) {
        constexpr double kTwoPi = 6.283185307179586;
        const double ang = static_cast<double>(pos[row]) * f;
        const double red = ang - rint(ang * (1.0 / kTwoPi)) * kTwoPi;
        float sn, cs;
        sincosf(static_cast<float>(red), &sn, &cs);
        s_cs[threadIdx.x] = make_float2(cs, sn);
    }
    __syncthreads();
    // heads: H query, Hk key (rotated; copied to k_new), then Hk value heads (copied to v_new)
    const int32_t heads = H + Hk + (v_new ? Hk : 0);
    const int32_t h0 = blockIdx.y * heads_per_block, h1 = min(heads, h0 + heads_per_block);
    const int32_t quads = half / 4, units = (h1 - h0) * quads;
    __nv_bfloat16 *x = qkv + static_cast<int64_t>(row) * nqkv;
    const int64_t kv_row = static_cast<int64_t>(row) * Hk * D;
    for (int32_t u = threadIdx.x; u < units; u += blockDim.x) {
        const int32_t hh = h0 + u / quads, j = (u - (u / quads) * quads) * 4;
        __nv_bfloat16 *e = x + hh * D + j;
        uint2 ra = *reinterpret_cast<const uint2 *>(e);
        uint2 rb = *reinterpret_cast<const uint2 *>(e + half);
        if (hh >= H + Hk) {  // a value head: copy
            __nv_bfloat16 *dst = v_new + kv_row + (hh - H - Hk) * D + j;
            *reinterpret_cast<uint2 *>(dst) = ra;
            *reinterpret_cast<uint2 *>(dst + half) = rb;
            continue;
        }
        __nv_bfloat16 *pa = reinterpret_cast<__nv_bfloat16 *>(&ra), *pb = reinterpret_cast<__nv_bfloat16 *>(&rb);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 c = s_cs[j + k];
            const float a = bf(pa[k]), b = bf(pb[k]);
            pa[k] = __float2bfloat16_rn(fmaf(a, c.x, -b * c.y));
            pb[k] = __float2bfloat16_rn(fmaf(b, c.x, a * c.y));
        }
        *reinterpret_cast<uint2 *>(e) = ra;
        *reinterpret_cast<uint2 *>(e + half) = rb;
        if (hh >= H && k_new) {
            __nv_bfloat16 *dst = k_new + kv_row + (hh - H) * D + j;
            *reinterpret_cast<uint2 *>(dst) = ra;
            *reinterpret_cast<uint2 *>(dst + half) = rb;
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Tree attention on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate)
// ---------------------------------------------------------------------------------------------
// CTA (request b, kv head hk, query tile, key split).  The query rows of (b, hk) are r = i * group
// + g (node i, query head hk * group + g); a warp owns 16 of them.  Keys: the P cached positions,
// then the n tree nodes (their rotated keys and values are columns of the qkv rows), in tiles of 64
// keys staged by cp.async in two stages.  Scores S = Q K^T / sqrt(D) stay in registers; a tree key
// counts for query node i when mask row i marks it; online softmax in fp32.  The probabilities go
// to the P V product as bf16 pairs p = hi + lo (hi = bf16(p), lo = bf16(p - hi)), which keeps them
// to ~2^-16 relative, as good as the fp32 sum they feed.  Splits of the key range write their
// unnormalised output, running max and sum; attention_combine_kernel merges them.
constexpr int kAttnKeys = 64;     // keys per tile
constexpr int kAttnMaxWarps = 4;  // 64 query rows per CTA

struct AttnArgs {
    int32_t B, n, P, H, Hk, nqkv, group, Mq, rows_cta, q_tiles, splits, tiles_per_split, W;
    const __nv_bfloat16 *qkv;      // [B*n][nqkv]: q (H*D), k (Hk*D), v (Hk*D), rotated
    const __nv_bfloat16 *k_cache;  // [B][P][Hk][D]
    const __nv_bfloat16 *v_cache;
    const uint32_t *mask;          // [B][n][W]
    __nv_bfloat16 *o;              // [B*n][H*D]
    float *part_o;                 // [splits][B*Hk*Mq][D]   (splits > 1)
    float2 *part_ml;               // [splits][B*Hk*Mq]      (running max, sum)
};

template <int D>
struct AttnShape {
    static constexpr int kRow = D + 8;  // smem row stride (elements): odd 16-byte stride, no ldmatrix conflicts
    static constexpr int kChunks = D / 8;
    static constexpr size_t smem_bytes(int rows_cta) {
        return (static_cast<size_t>(rows_cta) + 4 * kAttnKeys) * kRow * sizeof(__nv_bfloat16);
    }
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
    return *reinterpret_cast<uint32_t *>(&v);
}

// Key tile t of (request b, kv head hk) into `stage`: rows of K and V, cached positions first,
// then the tree nodes' rotated keys and values from the qkv rows; zero rows past the last key.
template <int D>
__device__ __forceinline__ void attn_load_tile(const AttnArgs &a, __nv_bfloat16 *sKV, int32_t t, int32_t stage,
                                               int32_t b, int32_t hk, int32_t total) {
    constexpr int kRow = AttnShape<D>::kRow, kChunks = AttnShape<D>::kChunks;
    __nv_bfloat16 *sK = sKV + (2 * stage) * kAttnKeys * kRow, *sV = sK + kAttnKeys * kRow;
    for (int32_t c = threadIdx.x; c < kAttnKeys * kChunks; c += blockDim.x) {
        const int32_t j = c / kChunks, ch = c - j * kChunks, key = t * kAttnKeys + j;
        const __nv_bfloat16 *kp = a.qkv, *vp = a.qkv;
        bool ok = true;
        if (key < a.P) {
            const int64_t off = ((static_cast<int64_t>(b) * a.P + key) * a.Hk + hk) * D + ch * 8;
            kp = a.k_cache + off;
            vp = a.v_cache + off;
        } else if (key < total) {
            const int64_t row = static_cast<int64_t>(b) * a.n + (key - a.P);
            kp = a.qkv + row * a.nqkv + (a.H + hk) * D + ch * 8;
            vp = a.qkv + row * a.nqkv + (a.H + a.Hk + hk) * D + ch * 8;
        } else {
            ok = false;  // past the last key: zero rows (finite values for the P V product)
        }
        cp_async16(sK + j * kRow + ch * 8, kp, ok);
        cp_async16(sV + j * kRow + ch * 8, vp, ok);
    }
}

template <int D, int KW>
__global__ void __launch_bounds__(kAttnMaxWarps * 32, 2) tree_attention_kernel(const AttnArgs a) {
    using S = AttnShape<D>;
    constexpr int kRow = S::kRow, kChunks = S::kChunks, kKS = D / 16, kNT = D / 8;
    constexpr int kSlice = kAttnKeys / KW, kSN = kSlice / 8, kPK = kSlice / 16;  // keys, n-tiles, k-steps
    extern __shared__ __align__(16) uint8_t attn_smem[];
    __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(attn_smem);
    __nv_bfloat16 *sKV = sQ + a.rows_cta * kRow;  // stage s: K at (2s) * 64 rows, V at (2s + 1) * 64 rows
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t nthreads = blockDim.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t qw = a.rows_cta / 16, qb = warp % qw, ks = warp / qw;  // query block, key slice
    const int32_t qt = blockIdx.x % a.q_tiles, pair = blockIdx.x / a.q_tiles;
    const int32_t b = pair / a.Hk, hk = pair - b * a.Hk;
    const int32_t r0 = qt * a.rows_cta;
    const int32_t total = a.P + a.n, num_tiles = (total + kAttnKeys - 1) / kAttnKeys;
    const int32_t t_begin = blockIdx.y * a.tiles_per_split;
    const int32_t t_end = min(num_tiles, t_begin + a.tiles_per_split);

    // query rows of this CTA (zero rows past Mq)
    for (int32_t c = threadIdx.x; c < a.rows_cta * kChunks; c += nthreads) {
        const int32_t r = c / kChunks, ch = c - r * kChunks, gr = r0 + r;
        const bool ok = gr < a.Mq;
        const int32_t i = ok ? gr / a.group : 0, g = ok ? gr - i * a.group : 0;
        const __nv_bfloat16 *src = a.qkv + static_cast<int64_t>(b * a.n + i) * a.nqkv + (hk * a.group + g) * D + ch * 8;
        cp_async16(sQ + r * kRow + ch * 8, src, ok);
    }
    auto load_tile = [&](int32_t t, int32_t stage) { attn_load_tile<D>(a, sKV, t, stage, b, hk, total); };
    load_tile(t_begin, 0);
    cp_async_commit();

    // this thread's two query rows (fragment rows g and g + 8 of its warp)
    const int32_t gq = lane >> 2, qd = lane & 3;
    const int32_t wrow0 = r0 + qb * 16;
    const bool warp_live = wrow0 < a.Mq;
    int32_t node[2];
    const uint32_t *mrow[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int32_t gr = wrow0 + gq + 8 * h;
        node[h] = gr < a.Mq ? gr / a.group : -1;
        mrow[h] = a.mask + static_cast<int64_t>(b * a.n + (node[h] < 0 ? 0 : node[h])) * a.W;
    }
    const float scale = 1.0f / sqrtf(static_cast<float>(D));
    uint32_t qf[kKS][4];
    float o[kNT][4];
#pragma unroll
    for (int j = 0; j < kNT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};

    for (int32_t t = t_begin; t < t_end; ++t) {
        const int32_t stage = (t - t_begin) & 1;
        if (t + 1 < t_end) load_tile(t + 1, stage ^ 1);
        cp_async_commit();
        cp_async_wait1();
        __syncthreads();
        if (warp_live) {
            const __nv_bfloat16 *sK = sKV + (2 * stage) * kAttnKeys * kRow + ks * kSlice * kRow;
            const __nv_bfloat16 *sV = sKV + (2 * stage + 1) * kAttnKeys * kRow + ks * kSlice * kRow;
            if (t == t_begin) {
#pragma unroll
                for (int k = 0; k < kKS; ++k)
                    ldsm_x4(qf[k], sQ + (qb * 16 + (lane & 15)) * kRow + k * 16 + (lane >> 4) * 8);
            }
            // S = Q K^T over this warp's slice of the tile: kSN n-tiles of 8 keys
            float s[kSN][4];
#pragma unroll
            for (int j = 0; j < kSN; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
#pragma unroll
            for (int k = 0; k < kKS; ++k) {
#pragma unroll
                for (int np = 0; np < kSN / 2; ++np) {
                    uint32_t kb[4];
                    ldsm_x4(kb, sK + (np * 16 + (lane & 7) + ((lane >> 4) << 3)) * kRow + k * 16 +
                                    ((lane >> 3) & 1) * 8);
                    mma_bf16(s[2 * np], qf[k], kb[0], kb[1]);
                    mma_bf16(s[2 * np + 1], qf[k], kb[2], kb[3]);
                }
            }
            // scale, mask, row max
            const int32_t key0 = t * kAttnKeys + ks * kSlice;
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < kSN; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = e >> 1;
                    const int32_t key = key0 + j * 8 + 2 * qd + (e & 1);
                    bool vis = node[h] >= 0 && key < total;
                    if (vis && key >= a.P) {
                        const int32_t tn = key - a.P;
                        vis = (mrow[h][tn >> 5] >> (tn & 31)) & 1u;
                    }
                    const float v = vis ? s[j][e] * scale : -INFINITY;
                    s[j][e] = v;
                    mx[h] = fmaxf(mx[h], v);
                }
            }
            float corr[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFullMask, mx[h], 1));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFullMask, mx[h], 2));
                const float nm = fmaxf(m_run[h], mx[h]);
                corr[h] = (m_run[h] == -INFINITY) ? 0.0f : expf(m_run[h] - nm);
                m_run[h] = nm;
                l_run[h] *= corr[h];
            }
#pragma unroll
            for (int j = 0; j < kNT; ++j) {
                o[j][0] *= corr[0];
                o[j][1] *= corr[0];
                o[j][2] *= corr[1];
                o[j][3] *= corr[1];
            }
            // probabilities (0 for hidden keys), then P V with P = hi + lo in bf16
#pragma unroll
            for (int j = 0; j < kSN; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = e >> 1;
                    const float p = (s[j][e] == -INFINITY) ? 0.0f : expf(s[j][e] - m_run[h]);
                    s[j][e] = p;
                    l_run[h] += p;
                }
            }
#pragma unroll
            for (int kk = 0; kk < kPK; ++kk) {  // 16 keys per k-step
                const float src[8] = {s[2 * kk][0], s[2 * kk][1], s[2 * kk][2], s[2 * kk][3],
                                      s[2 * kk + 1][0], s[2 * kk + 1][1], s[2 * kk + 1][2], s[2 * kk + 1][3]};
                float hi_f[8], lo_f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    hi_f[u] = __bfloat162float(__float2bfloat16_rn(src[u]));
                    lo_f[u] = src[u] - hi_f[u];
                }
                const uint32_t ph[4] = {pack_bf16(hi_f[0], hi_f[1]), pack_bf16(hi_f[2], hi_f[3]),
                                        pack_bf16(hi_f[4], hi_f[5]), pack_bf16(hi_f[6], hi_f[7])};
                const uint32_t pl[4] = {pack_bf16(lo_f[0], lo_f[1]), pack_bf16(lo_f[2], lo_f[3]),
                                        pack_bf16(lo_f[4], lo_f[5]), pack_bf16(lo_f[6], lo_f[7])};
#pragma unroll
                for (int np = 0; np < kNT / 2; ++np) {
                    uint32_t vb[4];
                    ldsm_x4_t(vb, sV + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kRow + np * 16 +
                                      (lane >> 4) * 8);
                    mma_bf16(o[2 * np], ph, vb[0], vb[1]);
                    mma_bf16(o[2 * np], pl, vb[0], vb[1]);
                    mma_bf16(o[2 * np + 1], ph, vb[2], vb[3]);
                    mma_bf16(o[2 * np + 1], pl, vb[2], vb[3]);
                }
            }
        }
        __syncthreads();  // the next iteration's loads overwrite this stage
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(kFullMask, l_run[h], 1);
        l_run[h] += __shfl_xor_sync(kFullMask, l_run[h], 2);
    }
    if constexpr (KW > 1) {
        // the key slices of each query block merge through shared memory (the stages are free now)
        float *mo = reinterpret_cast<float *>(sKV);                         // [KW * qw][16][D]
        float2 *mml = reinterpret_cast<float2 *>(mo + KW * qw * 16 * D);    // [KW * qw][16]
        const int32_t slot = ks * qw + qb;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int32_t row = gq + 8 * h;
#pragma unroll
            for (int j = 0; j < kNT; ++j)
                *reinterpret_cast<float2 *>(mo + (slot * 16 + row) * D + j * 8 + 2 * qd) =
                    make_float2(o[j][2 * h], o[j][2 * h + 1]);
            if (qd == 0) mml[slot * 16 + row] = make_float2(m_run[h], l_run[h]);
        }
        __syncthreads();
        if (ks != 0) return;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int32_t row = gq + 8 * h;
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < KW; ++k) M = fmaxf(M, mml[(k * qw + qb) * 16 + row].x);
            float wk[KW], L = 0.0f;
#pragma unroll
            for (int k = 0; k < KW; ++k) {
                const float2 ml = mml[(k * qw + qb) * 16 + row];
                wk[k] = (ml.x == -INFINITY) ? 0.0f : expf(ml.x - M);
                L += wk[k] * ml.y;
            }
#pragma unroll
            for (int j = 0; j < kNT; ++j) {
                float v0 = 0.0f, v1 = 0.0f;
#pragma unroll
                for (int k = 0; k < KW; ++k) {
                    const float2 p = *reinterpret_cast<const float2 *>(mo + ((k * qw + qb) * 16 + row) * D + j * 8 + 2 * qd);
                    v0 = fmaf(wk[k], p.x, v0);
                    v1 = fmaf(wk[k], p.y, v1);
                }
                o[j][2 * h] = v0;
                o[j][2 * h + 1] = v1;
            }
            m_run[h] = M;
            l_run[h] = L;
        }
    }
    if (!warp_live) return;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int32_t gr = wrow0 + gq + 8 * h;
        if (gr >= a.Mq) continue;
        if (a.splits == 1) {
            const int32_t i = node[h], g = gr - i * a.group, hq = hk * a.group + g;
            __nv_bfloat16 *orow = a.o + static_cast<int64_t>(b * a.n + i) * a.H * D + hq * D;
            const float inv = l_run[h] > 0.0f ? 1.0f / l_run[h] : 0.0f;
#pragma unroll
            for (int j = 0; j < kNT; ++j)
                *reinterpret_cast<__nv_bfloat162 *>(orow + j * 8 + 2 * qd) =
                    __floats2bfloat162_rn(o[j][2 * h] * inv, o[j][2 * h + 1] * inv);
        } else {
            const int64_t prow = static_cast<int64_t>(blockIdx.y) * a.B * a.Hk * a.Mq +
                                 static_cast<int64_t>(pair) * a.Mq + gr;
            float *po = a.part_o + prow * D;
#pragma unroll
            for (int j = 0; j < kNT; ++j)
                *reinterpret_cast<float2 *>(po + j * 8 + 2 * qd) = make_float2(o[j][2 * h], o[j][2 * h + 1]);
            if (qd == 0) a.part_ml[prow] = make_float2(m_run[h], l_run[h]);
        }
    }
}

// Few-query tree attention: at most 8 query rows per (request, kv head), e.g. one node per tree
// level and one query head per kv head.  The scores are formed transposed, S^T = K Q^T, with the 16
// keys of a warp's slice of the tile on the MMA's M side and the query rows on N = 8, and the
// output as O^T = V^T P^T with the head dims on M: no MMA row is padding, half the MMAs of the
// 16-row form.  A warp's probabilities move from the accumulator layout (key rows) to the
// B-operand layout (query columns) through a small shared-memory tile.  Tiles, stages, masking,
// the online softmax, the hi/lo split of P and the outputs are those of tree_attention_kernel.
constexpr int kFewWarps = 4;      // key slices of 16 keys per 64-key tile
constexpr int kFewPStride = 20;   // floats per row of the probability transpose: no bank conflicts

template <int D>
__global__ void __launch_bounds__(kFewWarps * 32, 3) tree_attention_few_kernel(const AttnArgs a) {
    using S = AttnShape<D>;
    constexpr int kRow = S::kRow, kChunks = S::kChunks, kKS = D / 16, kMT = D / 16;
    extern __shared__ __align__(16) uint8_t attn_smem[];
    __shared__ __align__(16) float sP[kFewWarps][8][kFewPStride];
    __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(attn_smem);  // 16 rows, the first Mq live
    __nv_bfloat16 *sKV = sQ + 16 * kRow;
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t ks = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t pair = blockIdx.x;  // one query tile
    const int32_t b = pair / a.Hk, hk = pair - b * a.Hk;
    const int32_t total = a.P + a.n, num_tiles = (total + kAttnKeys - 1) / kAttnKeys;
    const int32_t t_begin = blockIdx.y * a.tiles_per_split;
    const int32_t t_end = min(num_tiles, t_begin + a.tiles_per_split);

    for (int32_t c = threadIdx.x; c < 16 * kChunks; c += blockDim.x) {
        const int32_t r = c / kChunks, ch = c - r * kChunks;
        const bool ok = r < a.Mq;
        const int32_t i = ok ? r / a.group : 0, g = ok ? r - i * a.group : 0;
        const __nv_bfloat16 *src = a.qkv + static_cast<int64_t>(b * a.n + i) * a.nqkv + (hk * a.group + g) * D + ch * 8;
        cp_async16(sQ + r * kRow + ch * 8, src, ok);
    }
    attn_load_tile<D>(a, sKV, t_begin, 0, b, hk, total);
    cp_async_commit();

    // this thread's accumulator entries: keys (or head dims) gq and gq + 8, query columns 2 qd, 2 qd + 1
    const int32_t gq = lane >> 2, qd = lane & 3;
    int32_t node[2];
    const uint32_t *mrow[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int32_t q = 2 * qd + c;
        node[c] = q < a.Mq ? q / a.group : -1;
        mrow[c] = a.mask + static_cast<int64_t>(b * a.n + (node[c] < 0 ? 0 : node[c])) * a.W;
    }
    const float scale = 1.0f / sqrtf(static_cast<float>(D));
    uint32_t qb[kKS][2];
    float o[kMT][4];
#pragma unroll
    for (int j = 0; j < kMT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
    float (*pw)[kFewPStride] = sP[ks];

    for (int32_t t = t_begin; t < t_end; ++t) {
        const int32_t stage = (t - t_begin) & 1;
        if (t + 1 < t_end) attn_load_tile<D>(a, sKV, t + 1, stage ^ 1, b, hk, total);
        cp_async_commit();
        cp_async_wait1();
        __syncthreads();
        const __nv_bfloat16 *sK = sKV + (2 * stage) * kAttnKeys * kRow + ks * 16 * kRow;
        const __nv_bfloat16 *sV = sKV + (2 * stage + 1) * kAttnKeys * kRow + ks * 16 * kRow;
        if (t == t_begin) {  // Q^T as the B operand, two k-steps per load
#pragma unroll
            for (int k = 0; k < kKS; k += 2) {
                uint32_t r[4];
                ldsm_x4(r, sQ + (lane & 7) * kRow + (k + (lane >> 4)) * 16 + ((lane >> 3) & 1) * 8);
                qb[k][0] = r[0];
                qb[k][1] = r[1];
                qb[k + 1][0] = r[2];
                qb[k + 1][1] = r[3];
            }
        }
        // S^T over this warp's 16 keys; two accumulators over alternate k-steps
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int k = 0; k < kKS; ++k) {
            uint32_t ka[4];
            ldsm_x4(ka, sK + (lane & 15) * kRow + k * 16 + (lane >> 4) * 8);
            if (k & 1)
                mma_bf16(s2, ka, qb[k][0], qb[k][1]);
            else
                mma_bf16(s, ka, qb[k][0], qb[k][1]);
        }
        // scale, mask, column max over the warp's 16 keys
        const int32_t key0 = t * kAttnKeys + ks * 16;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = e & 1;
            const int32_t key = key0 + gq + 8 * (e >> 1);
            bool vis = node[c] >= 0 && key < total;
            if (vis && key >= a.P) {
                const int32_t tn = key - a.P;
                vis = (mrow[c][tn >> 5] >> (tn & 31)) & 1u;
            }
            const float v = vis ? (s[e] + s2[e]) * scale : -INFINITY;
            s[e] = v;
            mx[c] = fmaxf(mx[c], v);
        }
        float corr[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) mx[c] = fmaxf(mx[c], __shfl_xor_sync(kFullMask, mx[c], off));
            const float nm = fmaxf(m_run[c], mx[c]);
            corr[c] = (m_run[c] == -INFINITY) ? 0.0f : expf(m_run[c] - nm);
            m_run[c] = nm;
            l_run[c] *= corr[c];
        }
#pragma unroll
        for (int j = 0; j < kMT; ++j) {
            o[j][0] *= corr[0];
            o[j][1] *= corr[1];
            o[j][2] *= corr[0];
            o[j][3] *= corr[1];
        }
        // probabilities, then P (query rows) into the warp's transpose tile
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = e & 1;
            const float p = (s[e] == -INFINITY) ? 0.0f : expf(s[e] - m_run[c]);
            l_run[c] += p;
            pw[2 * qd + c][gq + 8 * (e >> 1)] = p;
        }
        __syncwarp();
        const float2 p_lo = *reinterpret_cast<const float2 *>(&pw[gq][2 * qd]);      // keys 2qd, 2qd+1
        const float2 p_hi = *reinterpret_cast<const float2 *>(&pw[gq][2 * qd + 8]);  // keys 2qd+8, 2qd+9
        const float src[4] = {p_lo.x, p_lo.y, p_hi.x, p_hi.y};
        float hi_f[4], lo_f[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            hi_f[u] = __bfloat162float(__float2bfloat16_rn(src[u]));
            lo_f[u] = src[u] - hi_f[u];
        }
        const uint32_t bh0 = pack_bf16(hi_f[0], hi_f[1]), bh1 = pack_bf16(hi_f[2], hi_f[3]);
        const uint32_t bl0 = pack_bf16(lo_f[0], lo_f[1]), bl1 = pack_bf16(lo_f[2], lo_f[3]);
        // O^T += V^T P^T, head dims on M
#pragma unroll
        for (int j = 0; j < kMT; ++j) {
            uint32_t va[4];
            ldsm_x4_t(va, sV + ((lane & 7) + (lane >> 4) * 8) * kRow + j * 16 + ((lane >> 3) & 1) * 8);
            mma_bf16(o[j], va, bh0, bh1);
            mma_bf16(o[j], va, bl0, bl1);
        }
        __syncthreads();  // the next iteration's loads overwrite this stage (and the transpose tile)
    }
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) l_run[c] += __shfl_xor_sync(kFullMask, l_run[c], off);

    // the four key slices merge through shared memory (the stages are free now)
    float *mo = reinterpret_cast<float *>(sKV);                       // [kFewWarps][8][D]
    float2 *mml = reinterpret_cast<float2 *>(mo + kFewWarps * 8 * D);  // [kFewWarps][8]
#pragma unroll
    for (int j = 0; j < kMT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            mo[(ks * 8 + 2 * qd + (e & 1)) * D + j * 16 + gq + 8 * (e >> 1)] = o[j][e];
    if (gq == 0) {
        mml[ks * 8 + 2 * qd] = make_float2(m_run[0], l_run[0]);
        mml[ks * 8 + 2 * qd + 1] = make_float2(m_run[1], l_run[1]);
    }
    __syncthreads();
    if (ks != 0) return;
    float wk[2][kFewWarps];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int32_t q = 2 * qd + c;
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kFewWarps; ++k) M = fmaxf(M, mml[k * 8 + q].x);
        float L = 0.0f;
#pragma unroll
        for (int k = 0; k < kFewWarps; ++k) {
            const float2 ml = mml[k * 8 + q];
            wk[c][k] = (ml.x == -INFINITY) ? 0.0f : expf(ml.x - M);
            L += wk[c][k] * ml.y;
        }
        m_run[c] = M;
        l_run[c] = L;
    }
#pragma unroll
    for (int j = 0; j < kMT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = e & 1;
            const int32_t q = 2 * qd + c, d = j * 16 + gq + 8 * (e >> 1);
            float v = 0.0f;
#pragma unroll
            for (int k = 0; k < kFewWarps; ++k) v = fmaf(wk[c][k], mo[(k * 8 + q) * D + d], v);
            o[j][e] = v;
        }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int32_t q = 2 * qd + c;
        if (q >= a.Mq) continue;
        if (a.splits == 1) {
            const int32_t i = node[c], g = q - i * a.group, hq = hk * a.group + g;
            __nv_bfloat16 *orow = a.o + static_cast<int64_t>(b * a.n + i) * a.H * D + hq * D;
            const float inv = l_run[c] > 0.0f ? 1.0f / l_run[c] : 0.0f;
#pragma unroll
            for (int j = 0; j < kMT; ++j) {
                orow[j * 16 + gq] = __float2bfloat16_rn(o[j][c] * inv);
                orow[j * 16 + gq + 8] = __float2bfloat16_rn(o[j][c + 2] * inv);
            }
        } else {
            const int64_t prow = static_cast<int64_t>(blockIdx.y) * a.B * a.Hk * a.Mq +
                                 static_cast<int64_t>(pair) * a.Mq + q;
            float *po = a.part_o + prow * D;
#pragma unroll
            for (int j = 0; j < kMT; ++j) {
                po[j * 16 + gq] = o[j][c];
                po[j * 16 + gq + 8] = o[j][c + 2];
            }
            if (gq == 0) a.part_ml[prow] = make_float2(m_run[c], l_run[c]);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Tree attention on the 5th-generation tensor cores (tcgen05, accumulators in tensor memory),
// for head_dim 64 or 128 and more than 64 query rows per (request, kv head).  CTA (request b,
// kv head hk, 128 query rows, key split), 6 warps:
//   warp 0     copies the key and value rows of each 64-key tile (cached keys, then the tree's
//              rotated keys and values from the qkv rows; zeros past the last key) in 16-byte
//              pieces (cp.async) into a ring of 3 stages, laid out 128-byte-swizzled with the
//              head dimension contiguous;
//   warp 1     one thread issues the MMAs:  S_t = Q K_t^T (M = 128 query rows, N = 64 keys,
//              K = D) into one of two TMEM score buffers, so the next tile's scores are formed
//              while this tile's softmax runs, and O += P_hi V_t + P_lo V_t (M = 128, N = D,
//              K = 64 keys; V is read as stored, the MN-major B operand) into a TMEM accumulator;
//   warps 2-5  one query row per thread (its TMEM lane): read the row of S_t, scale and mask it
//              (cached keys visible, tree keys by the node's mask row), keep a running max m and
//              sum l (base-2 exponentials), and write P = 2^(s - m) as bf16 hi + lo (the split of
//              the mma.sync kernels: ~2^-16 relative) into shared memory as the K-major A
//              operand.  O is rescaled in TMEM (read, multiplied, written back) only when a
//              tile's max exceeds m by more than 2^8: below that the terms stay in range, and O
//              and l keep the same m, so the output is unchanged.
// Output O / l in bf16, or with key splits the unnormalised O with m (natural log) and l for
// attention_combine_kernel.  Every wait is bounded (an expired wait ends the CTA's work; the
// copies and MMAs it started land before it exits).
// ---------------------------------------------------------------------------------------------
constexpr int kTcRows = 128;    // query rows per CTA: the MMA's M and the TMEM lanes
constexpr int kTcKeys = 64;     // keys per tile (the same tiles as kAttnKeys)
constexpr int kTcStages = 3;    // key/value tiles in flight
constexpr int kTcThreads = 320;  // warp 0 copies, warp 1 issues MMAs, warps 2-9 softmax
constexpr float kTcRescale = 8.0f;  // log2 of the growth allowed before O is rescaled
static_assert(kTcKeys == kAttnKeys, "key splits are planned in kAttnKeys tiles");

template <int D>
struct TcShape {
    static constexpr uint32_t kQBytes = kTcRows * D * 2;        // D / 64 blocks of [128 rows][64]
    static constexpr uint32_t kKVBytes = kTcKeys * D * 2;       // D / 64 blocks of [64 keys][64]
    static constexpr uint32_t kPBytes = kTcRows * kTcKeys * 2;  // [128 rows][64 keys], hi or lo
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kQBytes;
    static constexpr uint32_t kV = kK + kTcStages * kKVBytes;
    static constexpr uint32_t kP = kV + kTcStages * kKVBytes;
    static constexpr uint32_t kBar = kP + 2 * kPBytes;
    static constexpr size_t smem_bytes = kBar + 128 + 6 * kTcRows * 4 + 1024;  // barriers, row maxima and sums, alignment
};

struct TcBars {
    uint64_t kv_full[kTcStages];   // warp 0 -> MMA: tile copied
    uint64_t kv_empty[kTcStages];  // MMA (commit) -> warp 0: the tile's P V is done
    uint64_t s_full[2];            // MMA (commit) -> softmax: scores in the buffer
    uint64_t s_free[2];            // softmax (256) -> MMA: scores read
    uint64_t p_full;               // softmax (256) -> MMA: P written (and O rescaled)
    uint64_t o_done;               // MMA (commit) -> softmax: the tile's P V is done
    uint64_t q_ready;              // softmax (256) -> MMA: query rows copied
    uint64_t drain;                // unwinding after an expired wait
    uint32_t tmem_base;
    int32_t abort;
};

// Byte offset of 16-byte piece `chunk` (0..7) of row `row` in a 128-byte-swizzled block of
// 128-byte rows (the layout the tcgen05 descriptors with 128-byte swizzle read).
__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
static_assert(sizeof(TcBars) <= 128, "the row maxima follow the barriers");

// bar.sync over `n` threads of barrier `id` that also returns the OR of every thread's `pred`.
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    tree_attention_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                             const __grid_constant__ CUtensorMap tmap_qkv, const AttnArgs a) {
    using S = TcShape<D>;
    constexpr uint32_t kTmemCols = 256;  // S buffers at 0 and 64, O at 128
    extern __shared__ uint8_t tc_smem_raw[];
    const uint32_t raw_addr = smem_u32(tc_smem_raw);
    uint8_t *base = tc_smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    TcBars *bar = reinterpret_cast<TcBars *>(base + S::kBar);
    volatile int32_t *abort_flag = &bar->abort;
    const int32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t qt = blockIdx.x % a.q_tiles, pair = blockIdx.x / a.q_tiles;
    const int32_t b = pair / a.Hk, hk = pair - b * a.Hk;
    const int32_t total = a.P + a.n, num_tiles = (total + kTcKeys - 1) / kTcKeys;
    const int32_t t_begin = blockIdx.y * a.tiles_per_split;
    const int32_t T = max(0, min(num_tiles, t_begin + a.tiles_per_split) - t_begin);

    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&bar->kv_full[s], 1);
            mbar_init(&bar->kv_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar->s_full[i], 1);
            mbar_init(&bar->s_free[i], 256);
        }
        mbar_init(&bar->p_full, 256);
        mbar_init(&bar->o_done, 1);
        mbar_init(&bar->q_ready, 256);
        mbar_init(&bar->drain, 1);
        bar->abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&bar->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar->tmem_base;
    pdl_wait();  // qkv (rotated) and the caches come from earlier kernels

    if (warp == 0) {
        // ---------------- key/value copies ----------------
        // A tile of cached keys only: four (D = 128) or two tensor copies from the cache, counted
        // in bytes on the stage's barrier; a tile of tree keys only: the same from the qkv rows
        // (64 consecutive node rows; rows past the request's nodes are hidden keys, finite, or
        // zeros past the last row).  The one tile that holds both: 16-byte copies by the whole
        // warp, then one arrival.
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
            prefetch_tensormap(&tmap_qkv);
        }
        const uint64_t pol_qkv = policy_evict_last();  // the tree's keys are read by every query tile
        for (int32_t i = 0; i < T; ++i) {
            const int32_t st = i % kTcStages;
            if (i >= kTcStages) {
                int32_t ok = 1;
                if (lane == 0 && !mbar_wait(&bar->kv_empty[st], static_cast<uint32_t>(i / kTcStages - 1) & 1u, abort_flag)) {
                    ok = 0;
                    *abort_flag = 1;
                }
                if (!__shfl_sync(kFullMask, ok, 0)) break;
            }
            if (*abort_flag) break;
            const int32_t key0 = (t_begin + i) * kTcKeys;
            uint8_t *kd = base + S::kK + st * S::kKVBytes, *vd = base + S::kV + st * S::kKVBytes;
            if (key0 + kTcKeys <= a.P) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar->kv_full[st], 2u * S::kKVBytes);
#pragma unroll
                    for (int blk = 0; blk < D / 64; ++blk) {
                        tma_load_4d(kd + blk * (kTcKeys * 128), &tmap_k, &bar->kv_full[st], blk * 64, hk, key0, b);
                        tma_load_4d(vd + blk * (kTcKeys * 128), &tmap_v, &bar->kv_full[st], blk * 64, hk, key0, b);
                    }
                }
                __syncwarp();
                continue;
            }
            if (key0 >= a.P) {
                if (lane == 0) {
                    const int32_t y = b * a.n + (key0 - a.P);
                    mbar_arrive_expect_tx(&bar->kv_full[st], 2u * S::kKVBytes);
#pragma unroll
                    for (int blk = 0; blk < D / 64; ++blk) {
                        tma_load_2d(kd + blk * (kTcKeys * 128), &tmap_qkv, &bar->kv_full[st], (a.H + hk) * D + blk * 64,
                                    y, pol_qkv);
                        tma_load_2d(vd + blk * (kTcKeys * 128), &tmap_qkv, &bar->kv_full[st],
                                    (a.H + a.Hk + hk) * D + blk * 64, y, pol_qkv);
                    }
                }
                __syncwarp();
                continue;
            }
            fence_proxy_async_smem();  // the tensor cores' reads of this stage, before these writes
            for (int32_t c = lane; c < kTcKeys * (D / 8); c += 32) {
                const int32_t j = c / (D / 8), ch = c - j * (D / 8), key = key0 + j;
                const __nv_bfloat16 *kp = a.qkv, *vp = a.qkv;
                bool ok = true;
                if (key < a.P) {
                    const int64_t off = ((static_cast<int64_t>(b) * a.P + key) * a.Hk + hk) * D + ch * 8;
                    kp = a.k_cache + off;
                    vp = a.v_cache + off;
                } else if (key < total) {
                    const int64_t row = static_cast<int64_t>(b) * a.n + (key - a.P);
                    kp = a.qkv + row * a.nqkv + (a.H + hk) * D + ch * 8;
                    vp = a.qkv + row * a.nqkv + (a.H + a.Hk + hk) * D + ch * 8;
                } else {
                    ok = false;  // past the last key: zeros (P is 0 there; V must stay finite)
                }
                const uint32_t off = static_cast<uint32_t>(ch >> 3) * (kTcKeys * 128u) + sw128_off(j, ch & 7);
                cp_async16(kd + off, kp, ok);
                cp_async16(vd + off, vp, ok);
            }
            cp_async_commit();
            cp_async_wait_all();
            fence_proxy_async_smem();  // visible to the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->kv_full[st]);
        }
        cp_async_wait_all();
    } else if (warp == 1) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0 && T > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kTcRows, kTcKeys);
            constexpr uint32_t idesc_o = idesc_bf16_f32_bmn(kTcRows, D);
            const uint32_t q0 = smem_u32(base + S::kQ);
            auto issue_s = [&](int32_t i) -> bool {
                const int32_t st = i % kTcStages, sb = i & 1;
                if (!mbar_wait(&bar->kv_full[st], static_cast<uint32_t>(i / kTcStages) & 1u, abort_flag)) return false;
                if (i >= 2 && !mbar_wait(&bar->s_free[sb], static_cast<uint32_t>((i - 2) >> 1) & 1u, abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t k0 = smem_u32(base + S::kK + st * S::kKVBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t blk = kk >> 2, col = (kk & 3) * 32u;
                    mma_bf16_ss(tmem + sb * kTcKeys, sw128_kmajor_desc(q0 + blk * (kTcRows * 128u) + col),
                                sw128_kmajor_desc(k0 + blk * (kTcKeys * 128u) + col), idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar->s_full[sb]);
                return true;
            };
            bool ok = mbar_wait(&bar->q_ready, 0, abort_flag);
            if (ok) ok = issue_s(0);
            for (int32_t i = 0; i < T && ok; ++i) {
                if (i + 1 < T && !issue_s(i + 1)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(&bar->p_full, static_cast<uint32_t>(i) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int32_t st = i % kTcStages;
                const uint32_t v0 = smem_u32(base + S::kV + st * S::kKVBytes);
                const uint32_t ph = smem_u32(base + S::kP);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kTcKeys / 16; ++kk)  // 16 keys: two groups of 8 rows of V
                        mma_bf16_ss(tmem + 128u, sw128_kmajor_desc(ph + part * S::kPBytes + kk * 32u),
                                    sw128_desc(v0 + kk * 2048u, kTcKeys * 128u, 1024u), idesc_o,
                                    (i > 0 || part > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bar->o_done);
                mma_commit(&bar->kv_empty[st]);
            }
            if (!ok) *abort_flag = 1;
        }
        __syncwarp();
    } else {
        // ---------------- softmax and output: two threads a query row ----------------
        // warps 2-9: lane quarter w % 4 of TMEM (the rows), half h of each tile's keys and of O's
        // columns; the two halves of a row agree on its running max through shared memory
        const int32_t q = warp & 3, h = (warp - 2) >> 2, r = q * 32 + lane;
        const int32_t gr = qt * kTcRows + r;
        const bool live = gr < a.Mq;
        const int32_t node = live ? gr / a.group : 0, g = live ? gr - node * a.group : 0;
        {
            const __nv_bfloat16 *src = a.qkv + static_cast<int64_t>(b * a.n + node) * a.nqkv + (hk * a.group + g) * D;
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                const int ch = h * (D / 16) + c;
                cp_async16(base + S::kQ + (ch >> 3) * (kTcRows * 128u) + sw128_off(r, ch & 7), src + ch * 8, live);
            }
            cp_async_commit();
            cp_async_wait_all();
            fence_proxy_async_smem();
            mbar_arrive(&bar->q_ready);
        }
        const uint32_t *mrow = a.mask + static_cast<int64_t>(b * a.n + node) * a.W;
        const float sl2 = rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;  // 1/sqrt(D), base 2
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t o_cols = 128u + static_cast<uint32_t>(h * (D / 2));     // this half's columns of O
        uint8_t *ph = base + S::kP, *pl = ph + S::kPBytes;
        // [2 tiles][2 halves][128 rows] of row maxima, then [2 halves][128 rows] of row sums
        float *xmax = reinterpret_cast<float *>(base + S::kBar + 128);
        float m2 = -INFINITY, l = 0.0f;
        for (int32_t i = 0; i < T; ++i) {
            const int32_t sb = i & 1, key0 = (t_begin + i) * kTcKeys + h * 32;
            // an expired wait marks the CTA; the softmax warps leave the loop together, at the
            // barrier below, whose OR of the mark they all receive
            if (!mbar_wait(&bar->s_full[sb], static_cast<uint32_t>(i >> 1) & 1u, abort_flag)) *abort_flag = 1;
            __syncwarp();
            tc_fence_after();
            float s[32];
            {
                uint32_t v[32];
                tmem_ld_32(t_lane + sb * kTcKeys + h * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(v[j]);
            }
            tc_fence_before();
            mbar_arrive(&bar->s_free[sb]);
            // hidden keys to -inf (cached keys are visible, tree keys by the mask row: the 32
            // keys of this half tile span at most two of its words, read once)
            if (!live || key0 + 32 > a.P) {
                const int32_t t0 = key0 - a.P, first = max(t0, 0) >> 5;
                const uint32_t w0 = (live && first < a.W) ? mrow[first] : 0u;
                const uint32_t w1 = (live && first + 1 < a.W) ? mrow[first + 1] : 0u;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int32_t key = key0 + j, tn = t0 + j;
                    bool vis = live && key < total;
                    if (vis && tn >= 0) vis = (((tn >> 5) == first ? w0 : w1) >> (tn & 31)) & 1u;
                    if (!vis) s[j] = -INFINITY;
                }
            }
            float mq[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
            for (int j = 4; j < 32; ++j) mq[j & 3] = fmaxf(mq[j & 3], s[j]);
            xmax[((i & 1) * 2 + h) * kTcRows + r] = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            if (named_barrier_or(1, 256, *abort_flag != 0)) break;
            const float mx = fmaxf(xmax[((i & 1) * 2) * kTcRows + r], xmax[((i & 1) * 2 + 1) * kTcRows + r]) * sl2;
            const bool raise = mx > m2 + kTcRescale || (m2 == -INFINITY && mx > -INFINITY);
            float corr = 1.0f;
            if (raise) {
                corr = (m2 == -INFINITY) ? 0.0f : ex2_approx(m2 - mx);
                l *= corr;
                m2 = mx;
            }
            // P = 2^(s sl2 - m) as bf16 hi + lo, in registers before the previous P V is waited for
            const float mneg = (m2 == -INFINITY) ? 0.0f : -m2;  // hidden keys: 2^-inf = 0
            uint32_t hi[16], lo[16];
            float lsum[2] = {0.0f, 0.0f};
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float p0 = ex2_approx(fmaf(s[2 * u], sl2, mneg));
                const float p1 = ex2_approx(fmaf(s[2 * u + 1], sl2, mneg));
                lsum[u & 1] += p0 + p1;
                const __nv_bfloat162 hv = __floats2bfloat162_rn(p0, p1);
                const float2 hf = __bfloat1622float2(hv);
                const __nv_bfloat162 lv = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
                hi[u] = *reinterpret_cast<const uint32_t *>(&hv);
                lo[u] = *reinterpret_cast<const uint32_t *>(&lv);
            }
            l += lsum[0] + lsum[1];
            // the previous tile's P V is done: P's buffer is free and O holds every earlier tile
            if (i > 0 && !mbar_wait(&bar->o_done, static_cast<uint32_t>(i - 1) & 1u, abort_flag)) *abort_flag = 1;
            __syncwarp();
            tc_fence_after();
            if (i > 0 && __any_sync(kFullMask, raise && corr != 0.0f)) {
                // rescale this warp's rows of this half of O (a warp-wide TMEM round trip)
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t v[32];
                    tmem_ld_32(t_lane + o_cols + c * 32u, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * corr);
                    tmem_st_32(t_lane + o_cols + c * 32u, v);
                }
                tmem_wait_st();
            }
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                const uint32_t off = sw128_off(r, h * 4 + c8);
                *reinterpret_cast<uint4 *>(ph + off) = make_uint4(hi[4 * c8], hi[4 * c8 + 1], hi[4 * c8 + 2], hi[4 * c8 + 3]);
                *reinterpret_cast<uint4 *>(pl + off) = make_uint4(lo[4 * c8], lo[4 * c8 + 1], lo[4 * c8 + 2], lo[4 * c8 + 3]);
            }
            fence_proxy_async_smem();  // the writes above, before the MMA reads them
            tc_fence_before();         // and the rescale's TMEM stores
            mbar_arrive(&bar->p_full);
        }
        if (!*abort_flag && T > 0 && !mbar_wait(&bar->o_done, static_cast<uint32_t>(T - 1) & 1u, abort_flag))
            *abort_flag = 1;
        // the row's sum: both halves' shares (every softmax thread reaches this barrier)
        xmax[(4 + h) * kTcRows + r] = l;
        const bool stop = named_barrier_or(1, 256, *abort_flag != 0);
        const float lt = xmax[4 * kTcRows + r] + xmax[5 * kTcRows + r];
        __syncwarp();
        if (!stop) {
            tc_fence_after();
            const int64_t prow = static_cast<int64_t>(blockIdx.y) * a.B * a.Hk * a.Mq + static_cast<int64_t>(pair) * a.Mq + gr;
            __nv_bfloat16 *orow = a.o + static_cast<int64_t>(b * a.n + node) * a.H * D + (hk * a.group + g) * D + h * (D / 2);
            const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t v[32];
                tmem_ld_32(t_lane + o_cols + c * 32u, v);
                tmem_wait_ld();
                if (!live) continue;
                if (a.splits == 1) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 pk;
                        uint32_t *pw = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const __nv_bfloat162 hv = __floats2bfloat162_rn(__uint_as_float(v[e + 2 * u]) * inv,
                                                                            __uint_as_float(v[e + 2 * u + 1]) * inv);
                            pw[u] = *reinterpret_cast<const uint32_t *>(&hv);
                        }
                        *reinterpret_cast<uint4 *>(orow + c * 32 + e) = pk;
                    }
                } else {
                    float *po = a.part_o + prow * D + h * (D / 2) + c * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(po + e) =
                            make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                        __uint_as_float(v[e + 3]));
                }
            }
            if (live && a.splits > 1 && h == 0) a.part_ml[prow] = make_float2(m2 * 0.6931471805599453f, lt);
        }
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_flag && warp == 1 && lane == 0) {
        // let every MMA this CTA issued land before its memory is handed on
        mma_commit(&bar->drain);
        mbar_wait(&bar->drain, 0, nullptr);
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merges the key splits of each query row: o = sum_s w_s O_s / sum_s w_s l_s with
// w_s = exp(m_s - max_s m_s) (0 for a split that saw no visible key).  A warp per query row: lane
// s reads split s's (max, sum) (at most 32 splits), then each lane sums 4 output columns.
constexpr int kCombineRows = 4;

__global__ void __launch_bounds__(kCombineRows * 32) attention_combine_kernel(const AttnArgs a, int32_t D) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int64_t rows = static_cast<int64_t>(a.B) * a.Hk * a.Mq;
    const int64_t prow = static_cast<int64_t>(blockIdx.x) * kCombineRows + (threadIdx.x >> 5);
    if (prow >= rows) return;
    const int32_t lane = threadIdx.x & 31;
    const float2 ml = lane < a.splits ? a.part_ml[lane * rows + prow] : make_float2(-INFINITY, 0.0f);
    float M = ml.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    const float wgt = (ml.x == -INFINITY) ? 0.0f : expf(ml.x - M);
    float L = wgt * ml.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFullMask, L, off);
    const float scale_s = L > 0.0f ? wgt / L : 0.0f;  // lane s: weight of split s in the output
    const int32_t pair = static_cast<int32_t>(prow / a.Mq), gr = static_cast<int32_t>(prow - static_cast<int64_t>(pair) * a.Mq);
    const int32_t b = pair / a.Hk, hk = pair - b * a.Hk, i = gr / a.group, g = gr - i * a.group;
    __nv_bfloat16 *orow = a.o + static_cast<int64_t>(b * a.n + i) * a.H * D + (hk * a.group + g) * D;
    for (int32_t c = lane * 4; c < D; c += 128) {
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int32_t s = 0; s < a.splits; ++s) {
            const float w = __shfl_sync(kFullMask, scale_s, s);
            if (w == 0.0f) continue;
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.part_o + (s * rows + prow) * D + c));
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(orow + c) = pk;
    }
}

// h1 = bf16(x + y) (x bf16, y fp32) and r = bf16(h1 * rsqrt(mean(h1^2) + eps) * w), one block per
// row, 8 elements per access (h a multiple of 8).
__global__ void __launch_bounds__(256) add_rmsnorm_kernel(const __nv_bfloat16 *x, const float *y,
                                                          const __nv_bfloat16 *w, __nv_bfloat16 *h1,
                                                          __nv_bfloat16 *r, int32_t h, float eps) {
    __shared__ float red[8];
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * h;
    float ss = 0.0f;
    for (int32_t e = threadIdx.x * 8; e < h; e += blockDim.x * 8) {
        const uint4 xv = *reinterpret_cast<const uint4 *>(x + base + e);
        const float4 y0 = *reinterpret_cast<const float4 *>(y + base + e);
        const float4 y1 = *reinterpret_cast<const float4 *>(y + base + e + 4);
        const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(&xv);
        const float yy[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        uint4 hv;
        __nv_bfloat16 *hb = reinterpret_cast<__nv_bfloat16 *>(&hv);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            hb[k] = __float2bfloat16_rn(bf(xb[k]) + yy[k]);
            const float v = bf(hb[k]);
            ss = fmaf(v, v, ss);
        }
        *reinterpret_cast<uint4 *>(h1 + base + e) = hv;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(kFullMask, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();  // also orders this block's h1 stores before the reads below
    float tot = 0.0f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) tot += red[i];
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(h) + eps);
    for (int32_t e = threadIdx.x * 8; e < h; e += blockDim.x * 8) {
        const uint4 hv = *reinterpret_cast<const uint4 *>(h1 + base + e);
        const uint4 wv = *reinterpret_cast<const uint4 *>(w + e);
        const __nv_bfloat16 *hb = reinterpret_cast<const __nv_bfloat16 *>(&hv);
        const __nv_bfloat16 *wb = reinterpret_cast<const __nv_bfloat16 *>(&wv);
        uint4 ov;
        __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(&ov);
#pragma unroll
        for (int k = 0; k < 8; ++k) ob[k] = __float2bfloat16_rn(bf(hb[k]) * inv * bf(wb[k]));
        *reinterpret_cast<uint4 *>(r + base + e) = ov;
    }
}

// out = bf16(x + y) element-wise (x bf16, y fp32), 8 elements per access (count a multiple of 8).
__global__ void __launch_bounds__(256) residual_kernel(const __nv_bfloat16 *x, const float *y, __nv_bfloat16 *out,
                                                       int64_t count) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < count;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x * 8) {
        const uint4 xv = *reinterpret_cast<const uint4 *>(x + i);
        const float4 y0 = *reinterpret_cast<const float4 *>(y + i);
        const float4 y1 = *reinterpret_cast<const float4 *>(y + i + 4);
        const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(&xv);
        const float yy[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        uint4 ov;
        __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(&ov);
#pragma unroll
        for (int k = 0; k < 8; ++k) ob[k] = __float2bfloat16_rn(bf(xb[k]) + yy[k]);
        *reinterpret_cast<uint4 *>(out + i) = ov;
    }
}

// a = bf16(silu(g) * u), g and u the two halves of each gu row; 8 elements per access (I a
// multiple of 8).
__global__ void __launch_bounds__(256) swiglu_kernel(const __nv_bfloat16 *gu, __nv_bfloat16 *act, int32_t I,
                                                     int64_t rows) {
    pdl_launch_dependents();  // dependents still wait for this grid to finish
    pdl_wait();
    const int32_t per_row = I / 8;
    const int64_t units = rows * per_row;
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = u / per_row, e = (u - row * per_row) * 8;
        const uint4 gv = *reinterpret_cast<const uint4 *>(gu + row * 2 * I + e);
        const uint4 uv = *reinterpret_cast<const uint4 *>(gu + row * 2 * I + I + e);
        const __nv_bfloat16 *gb = reinterpret_cast<const __nv_bfloat16 *>(&gv);
        const __nv_bfloat16 *ub = reinterpret_cast<const __nv_bfloat16 *>(&uv);
        uint4 ov;
        __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(&ov);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float g = bf(gb[k]);
            ob[k] = __float2bfloat16_rn(g / (1.0f + expf(-g)) * bf(ub[k]));
        }
        *reinterpret_cast<uint4 *>(act + row * I + e) = ov;
    }
}

}  // namespace

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
namespace {

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct DecoderLayout {
    size_t qkv, o, y, h1, r, gu, act, counters, partials, part_o, part_ml, total;
};

constexpr int32_t kAttnMaxSplits = 32;

// Attention launch shape: query rows per CTA (16 per warp), query tiles, and the largest key
// split count (enough CTAs for two per SM when (request, kv head, query tile) alone are fewer).
struct AttnPlan {
    int32_t group, Mq, qw, kw, warps, rows_cta, q_tiles, splits_max;
    bool few;  // at most 8 query rows per (request, kv head): tree_attention_few_kernel
    bool tc;   // head_dim 64 or 128 and more than 64 query rows: tree_attention_tc_kernel
};

AttnPlan attn_plan(const eagle_decoder_layer_weights *w, int32_t batch, int32_t nodes, int32_t sms) {
    AttnPlan p{};
    p.group = w->heads / w->kv_heads;
    p.Mq = nodes * p.group;
    p.qw = std::min(kAttnMaxWarps, (p.Mq + 15) / 16);          // warps over query rows
    p.kw = p.qw == 1 ? 4 : (p.qw == 2 ? 2 : 1);                // warps over each key tile
    p.warps = p.qw * p.kw;
    p.rows_cta = p.qw * 16;
    p.q_tiles = (p.Mq + p.rows_cta - 1) / p.rows_cta;
    p.few = p.Mq <= 8;  // one warp's 16-row tile would be half padding: the transposed kernel
    p.tc = (w->head_dim == 64 || w->head_dim == 128) && p.Mq > 64;
    if (p.tc) {
        p.rows_cta = kTcRows;
        p.q_tiles = (p.Mq + kTcRows - 1) / kTcRows;
    }
    const int64_t ctas = static_cast<int64_t>(batch) * w->kv_heads * p.q_tiles;
    p.splits_max = ctas >= 2 * sms ? 1 : static_cast<int32_t>(std::min<int64_t>(kAttnMaxSplits, (2 * sms + ctas - 1) / ctas));
    return p;
}

// Key splits for `prefix` cached keys: at most splits_max, at least two key tiles per split.
void attn_splits(const AttnPlan &p, int32_t prefix, int32_t nodes, int32_t *splits, int32_t *tiles_per_split) {
    const int32_t tiles = (prefix + nodes + kAttnKeys - 1) / kAttnKeys;
    int32_t s = std::max(1, std::min(p.splits_max, tiles / 2));
    const int32_t tps = (tiles + s - 1) / s;
    *tiles_per_split = tps;
    *splits = (tiles + tps - 1) / tps;
}

bool decoder_dims_ok(const eagle_decoder_layer_weights *w) {
    if (!w || w->hidden < 8 || w->hidden % 8 || w->heads < 1 || w->kv_heads < 1 || w->heads % w->kv_heads) return false;
    if (w->head_dim < 32 || w->head_dim > kMaxHeadDim || w->head_dim % 32) return false;
    if (w->inter < 8 || w->inter % 8) return false;
    if (!(w->rope_theta > 0.0f) || !(w->rms_eps >= 0.0f)) return false;
    return true;
}

DecoderLayout decoder_layout(const eagle_decoder_layer_weights *w, int32_t batch, int32_t nodes, int32_t sms) {
    const int64_t rows = static_cast<int64_t>(batch) * nodes;
    const int64_t h = w->hidden, nq = static_cast<int64_t>(w->heads) * w->head_dim;
    const int64_t nk = static_cast<int64_t>(w->kv_heads) * w->head_dim, I = w->inter;
    const int64_t nqkv = nq + 2 * nk;
    DecoderLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + (bytes ? bytes : 1));
        return at;
    };
    const int32_t chunk = static_cast<int32_t>(std::min<int64_t>(rows, kLinearMaxRows));
    const int32_t widest = static_cast<int32_t>(std::max<int64_t>(std::max(nqkv, h), 2 * I));
    L.counters = take(linear_counters_bytes(widest, static_cast<int32_t>(rows)));
    L.partials = take(linear_partials_bytes(sms, linear_n_tile(chunk)));
    L.qkv = take(static_cast<size_t>(rows) * nqkv * 2);
    L.o = take(static_cast<size_t>(rows) * nq * 2);
    L.y = take(static_cast<size_t>(rows) * h * 4);
    L.h1 = take(static_cast<size_t>(rows) * h * 2);
    L.r = take(static_cast<size_t>(rows) * h * 2);
    L.gu = take(static_cast<size_t>(rows) * 2 * I * 2);
    L.act = take(static_cast<size_t>(rows) * I * 2);
    const AttnPlan ap = attn_plan(w, batch, nodes, sms);
    const size_t prows = ap.splits_max > 1 ? static_cast<size_t>(ap.splits_max) * batch * w->kv_heads * ap.Mq : 0;
    L.part_o = take(prows * w->head_dim * 4);
    L.part_ml = take(prows * 8);
    L.total = o;
    return L;
}

int32_t sms_now() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Y = X W^T over all `rows` rows in one launch: every weight byte is read from HBM once for all
// row chunks (a weight tile's chunks are consecutive units of the split).
cudaError_t gemm_rows(const void *W, int32_t M, int32_t K, const void *X, int32_t rows, void *Y, int32_t out_bf16,
                      float *partials, int32_t *counters, int32_t sms, cudaStream_t st) {
    LinearPlan p;
    if (!plan_linear_bf16(&p, W, K, M, K, X, K, rows, nullptr, Y, M, out_bf16, partials, counters, nullptr, sms))
        return cudaErrorInvalidValue;
    return launch_linear_bf16(p, st);
}

template <int D>
cudaError_t set_attention_smem() {
    const int32_t bytes = static_cast<int32_t>(AttnShape<D>::smem_bytes(kAttnMaxWarps * 16));
    cudaError_t e = cudaFuncSetAttribute(tree_attention_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tree_attention_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tree_attention_kernel<D, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tree_attention_few_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int32_t>(AttnShape<D>::smem_bytes(16)));
    if constexpr (D == 64 || D == 128) {
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tree_attention_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int32_t>(TcShape<D>::smem_bytes));
    }
    return e;
}

template <int D>
cudaError_t launch_attention(const AttnPlan &ap, dim3 grid, const AttnArgs &aa, const CUtensorMap &tk,
                             const CUtensorMap &tv, const CUtensorMap &tq, cudaStream_t st) {
    if constexpr (D == 64 || D == 128) {
        if (ap.tc)
            return launch_pdl(tree_attention_tc_kernel<D>, grid, dim3(kTcThreads), TcShape<D>::smem_bytes, st, tk, tv,
                              tq, aa);
    }
    const dim3 block(ap.warps * 32);
    const size_t smem = AttnShape<D>::smem_bytes(ap.rows_cta);
    if (ap.few) return launch_pdl(tree_attention_few_kernel<D>, grid, block, smem, st, aa);
    if (ap.kw == 4) return launch_pdl(tree_attention_kernel<D, 4>, grid, block, smem, st, aa);
    if (ap.kw == 2) return launch_pdl(tree_attention_kernel<D, 2>, grid, block, smem, st, aa);
    return launch_pdl(tree_attention_kernel<D, 1>, grid, block, smem, st, aa);
}

std::mutex g_prep_mu;
bool g_prepared[64] = {};

cudaError_t prepare_once(int dev) {
    std::lock_guard<std::mutex> lock(g_prep_mu);
    if (g_prepared[dev]) return cudaSuccess;
    cudaError_t e = prepare_kernels();
    if (e == cudaSuccess) e = set_attention_smem<32>();
    if (e == cudaSuccess) e = set_attention_smem<64>();
    if (e == cudaSuccess) e = set_attention_smem<96>();
    if (e == cudaSuccess) e = set_attention_smem<128>();
    if (e == cudaSuccess) g_prepared[dev] = true;
    return e;
}

}  // namespace
}  // namespace eagle

extern "C" {

size_t eagle_decoder_layer_workspace_bytes(const eagle_decoder_layer_weights *w, int32_t batch, int32_t nodes) {
    if (!eagle::decoder_dims_ok(w) || batch < 1 || nodes < 1) return 0;
    const int32_t sms = eagle::sms_now();
    if (sms < 1) return 0;
    return eagle::decoder_layout(w, batch, nodes, sms).total;
}

eagle_status eagle_decoder_layer(const eagle_decoder_layer_weights *w, int32_t batch, int32_t nodes, int32_t prefix,
                                 const void *d_x, const void *d_k_cache, const void *d_v_cache,
                                 const int32_t *d_positions, const uint32_t *d_mask, void *d_out, void *d_k_new,
                                 void *d_v_new, void *d_ws, size_t ws_bytes, eagle_stream_t stream) {
    using namespace eagle;
    NvtxRange nvtx_range("eagle_decoder_layer");
    if (!decoder_dims_ok(w) || batch < 0 || nodes < 1 || nodes > kMaxCandidates + 1 || prefix < 0)
        return EAGLE_ERR_INVALID_ARG;
    if (batch == 0) return EAGLE_OK;
    if (!w->w_qkv || !w->w_o || !w->w_norm || !w->w_gu || !w->w_d || !d_x || !d_positions || !d_mask || !d_out ||
        !d_ws)
        return EAGLE_ERR_INVALID_ARG;
    if (prefix > 0 && (!d_k_cache || !d_v_cache)) return EAGLE_ERR_INVALID_ARG;
    if ((d_k_new == nullptr) != (d_v_new == nullptr)) return EAGLE_ERR_INVALID_ARG;
    const void *ptrs[] = {w->w_qkv, w->w_o, w->w_norm, w->w_gu, w->w_d, d_x, d_out, d_k_cache, d_v_cache,
                          d_k_new, d_v_new};
    for (const void *p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) & 15u) return EAGLE_ERR_INVALID_ARG;  // null passes
    if (reinterpret_cast<uintptr_t>(d_ws) & 255u) return EAGLE_ERR_INVALID_ARG;
    const int32_t sms = sms_now();
    int dev = 0;
    if (sms < 1 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return EAGLE_ERR_CUDA;
    if (prepare_once(dev) != cudaSuccess) return EAGLE_ERR_CUDA;
    const int32_t rows = batch * nodes;
    const DecoderLayout L = decoder_layout(w, batch, nodes, sms);
    if (ws_bytes < L.total) return EAGLE_ERR_INVALID_ARG;
    uint8_t *ws = reinterpret_cast<uint8_t *>(d_ws);
    auto at = [&](size_t off) { return ws + off; };
    float *partials = reinterpret_cast<float *>(at(L.partials));
    int32_t *counters = reinterpret_cast<int32_t *>(at(L.counters));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int32_t h = w->hidden, H = w->heads, Hk = w->kv_heads, D = w->head_dim, I = w->inter;
    const int32_t nq = H * D, nk = Hk * D, nqkv = nq + 2 * nk;
    auto *qkv = reinterpret_cast<__nv_bfloat16 *>(at(L.qkv));
    auto *o = reinterpret_cast<__nv_bfloat16 *>(at(L.o));
    auto *y = reinterpret_cast<float *>(at(L.y));
    auto *h1 = reinterpret_cast<__nv_bfloat16 *>(at(L.h1));
    auto *r = reinterpret_cast<__nv_bfloat16 *>(at(L.r));
    auto *gu = reinterpret_cast<__nv_bfloat16 *>(at(L.gu));
    auto *act = reinterpret_cast<__nv_bfloat16 *>(at(L.act));
    const int64_t hcount = static_cast<int64_t>(rows) * h;
    const int32_t eblocks = static_cast<int32_t>(std::min<int64_t>(4 * sms, (hcount / 8 + 255) / 256));
#define DEC_CUDA(expr)                              \
    do {                                            \
        if ((expr) != cudaSuccess) return EAGLE_ERR_CUDA; \
    } while (0)
    // projections of every node, rotated
    DEC_CUDA(gemm_rows(w->w_qkv, nqkv, h, d_x, rows, qkv, 1, partials, counters, sms, st));
    // rotation (one block per row, heads split over more blocks when rows are few); the tree's
    // rotated keys and values go out to k_new / v_new here
    const int32_t heads_all = H + Hk + (d_v_new ? Hk : 0);
    int32_t hsplit = rows >= 2 * sms ? 1 : std::min((2 * sms + rows - 1) / rows, std::max(1, heads_all / 8));
    const int32_t heads_per_block = (heads_all + hsplit - 1) / hsplit;
    hsplit = (heads_all + heads_per_block - 1) / heads_per_block;
    DEC_CUDA(launch_pdl(rope_kernel, dim3(rows, hsplit), dim3(256), 0, st, qkv, nqkv, H, Hk, heads_per_block, D,
                        d_positions, static_cast<double>(w->rope_theta), reinterpret_cast<__nv_bfloat16 *>(d_k_new),
                        reinterpret_cast<__nv_bfloat16 *>(d_v_new)));
    // tree attention over the cache and the tree
    const AttnPlan ap = attn_plan(w, batch, nodes, sms);
    int32_t splits = 1, tps = 1;
    attn_splits(ap, prefix, nodes, &splits, &tps);
    AttnArgs aa{batch, nodes, prefix, H, Hk, nqkv, ap.group, ap.Mq, ap.rows_cta, ap.q_tiles, splits, tps,
                (nodes + 31) / 32, qkv, reinterpret_cast<const __nv_bfloat16 *>(d_k_cache),
                reinterpret_cast<const __nv_bfloat16 *>(d_v_cache), d_mask, o,
                reinterpret_cast<float *>(at(L.part_o)), reinterpret_cast<float2 *>(at(L.part_ml))};
    const dim3 agrid(batch * Hk * ap.q_tiles, splits);
    // the tensor-core kernel reads whole tiles of cached keys by tensor copies
    CUtensorMap tk{}, tv{}, tq{};
    if (ap.tc && prefix > 0 &&
        (!encode_kv_cache_map(&tk, d_k_cache, batch, prefix, Hk, D) ||
         !encode_kv_cache_map(&tv, d_v_cache, batch, prefix, Hk, D)))
        return EAGLE_ERR_CUDA;
    if (ap.tc && !encode_bf16_rows_map(&tq, qkv, static_cast<uint64_t>(nqkv), static_cast<uint64_t>(rows),
                                       static_cast<uint64_t>(nqkv), 64, kTcKeys))
        return EAGLE_ERR_CUDA;
    switch (D) {
        case 32: DEC_CUDA(launch_attention<32>(ap, agrid, aa, tk, tv, tq, st)); break;
        case 64: DEC_CUDA(launch_attention<64>(ap, agrid, aa, tk, tv, tq, st)); break;
        case 96: DEC_CUDA(launch_attention<96>(ap, agrid, aa, tk, tv, tq, st)); break;
        default: DEC_CUDA(launch_attention<128>(ap, agrid, aa, tk, tv, tq, st)); break;
    }
    if (splits > 1)
        DEC_CUDA(launch_pdl(attention_combine_kernel, dim3((batch * Hk * ap.Mq + kCombineRows - 1) / kCombineRows),
                            dim3(kCombineRows * 32), 0, st, aa, D));
    // output projection, residual and post-attention RMSNorm
    DEC_CUDA(gemm_rows(w->w_o, h, nq, o, rows, y, 0, partials, counters, sms, st));
    DEC_CUDA(launch_pdl(add_rmsnorm_kernel, dim3(rows), dim3(256), 0, st, reinterpret_cast<const __nv_bfloat16 *>(d_x),
                        static_cast<const float *>(y), reinterpret_cast<const __nv_bfloat16 *>(w->w_norm), h1, r, h,
                        w->rms_eps));
    // SwiGLU MLP and residual
    DEC_CUDA(gemm_rows(w->w_gu, 2 * I, h, r, rows, gu, 1, partials, counters, sms, st));
    const int64_t aunits = static_cast<int64_t>(rows) * (I / 8);
    DEC_CUDA(launch_pdl(swiglu_kernel, dim3(static_cast<int32_t>(std::min<int64_t>(4 * sms, (aunits + 255) / 256))),
                        dim3(256), 0, st, static_cast<const __nv_bfloat16 *>(gu), act, I, static_cast<int64_t>(rows)));
    DEC_CUDA(gemm_rows(w->w_d, h, I, act, rows, y, 0, partials, counters, sms, st));
    DEC_CUDA(launch_pdl(residual_kernel, dim3(eblocks), dim3(256), 0, st, static_cast<const __nv_bfloat16 *>(h1),
                        static_cast<const float *>(y), reinterpret_cast<__nv_bfloat16 *>(d_out), hcount));
#undef DEC_CUDA
    return EAGLE_OK;
}

}  // extern "C"
