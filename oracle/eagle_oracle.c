/*
 * eagle_oracle.c - CPU oracle of one EAGLE / EAGLE-2 dynamic draft-tree step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file restates the method as plain, slow loops so that a
 * reader can check it against the pages by eye.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it; the product (the CUDA library) never does, and the two
 * share no code, header, table or helper.  The only thing both sides consume is the seeded
 * input generator, which holds none of the method's arithmetic.
 *
 * Sources (web pages, cited by title and section):
 *   [notes04]  "EAGLE 推测解码为什么比 Medusa 快？（含 EAGLE-2 动态草稿树）"
 *              (zzszmyf.github.io speculative-decoding notes, chapter 04)
 *   [tomjerr]  "(EAGLE 1) EAGLE: Speculative Sampling Requires Rethinking Feature Uncertainty"
 *              (tom-jerr.github.io paper reading)
 *   [zdszero]  Medusa -> EAGLE -> EAGLE-2 notes (zdszero.github.io, spec_medusa_eagle), with its
 *              sections "draft 结构", "EAGLE-2：树的形状应该跟着上下文变" and "在 SGLang 里"
 *   [jsqmd]    "投机解码：从eagle1到dflash" (jsqmd.com), section "二、EAGLE-2"
 *
 * Arithmetic contract (the pages fix none; these are the readings the test suite relies on):
 *   - every dot product accumulates in fp32, terms added in ascending index order, each product
 *     rounded to fp32 before its add (the file is built with -ffp-contract=off, so no host fuses
 *     them into an FMA);
 *   - bf16 inputs are widened exactly to fp32 (a bf16 is the upper half of a binary32);
 *   - for bf16 configurations the FC output is rounded once to bf16, round-to-nearest-even;
 *   - path scores are kept as fp32 logs, S(child) = fl(S(parent) + logp(child)): a monotone
 *     restatement of the product of confidences in [notes04] §10.3;
 *   - every ranking breaks ties toward the lowest index (token id, or candidate id, which is
 *     level-major so a shallower node wins a tie, as [notes04] §10.3 property 2 asks).
 *
 * Parity status of each function: pinned by tests/test_oracle_*.py (see the header of each
 * function for its pin).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_TREE 2  /* a kept node's parent was not kept: the connectivity property failed */
#define ORC_ERR_NOMEM 3

/* ------------------------------------------------------------------------------------------ */
/* Number formats                                                                             */
/* ------------------------------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of an IEEE-754 binary32; widening is exact. */
float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to bf16, to nearest, ties to even.  NaN stays a (quiet) NaN.
 * Pin: equals torch's float32 -> bfloat16 conversion on every tested bit pattern. */
uint16_t orc_f32_to_bf16(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static float load_elem(const void *p, int32_t is_bf16, int64_t i) {
    return is_bf16 ? orc_bf16_to_f32(((const uint16_t *)p)[i]) : ((const float *)p)[i];
}

int32_t orc_num_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int32_t n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------------------------ */
/* One draft row: FC then LM head                                                             */
/* ------------------------------------------------------------------------------------------ */

/* [notes04] §4.1 and [zdszero] "draft 结构": the draft input is the concatenation
 * [f || e(t)] in R^{2h} of a feature and the embedding of the (shifted) next token; an FC
 * (2h -> h, with bias) maps it back to h.  The decoder layer that follows the FC on the pages
 * is taken as the identity here (spec scope: FC then LM head).
 *   w_fc : [h][2h] row-major; columns 0..h-1 act on the feature, h..2h-1 on e(t)
 *   b_fc : [h] or NULL
 *   feat : [h] fp32 (already widened)
 *   emb  : [V][h] embedding table; row `tok` is e(t)
 *   fhat : [h] out, fp32 (holding a bf16 value when is_bf16)
 * Pin: float64 matrix product of the same widened inputs, within the fp32 dot-product bound. */
void orc_fc_row(int32_t h, int32_t is_bf16, const void *w_fc, const void *b_fc,
                const float *feat, const void *emb, int32_t tok, float *fhat) {
#pragma omp parallel for schedule(static)
    for (int32_t o = 0; o < h; ++o) {
        float acc = 0.0f;
        for (int32_t i = 0; i < 2 * h; ++i) {
            float x = (i < h) ? feat[i] : load_elem(emb, is_bf16, (int64_t)tok * h + (i - h));
            float w = load_elem(w_fc, is_bf16, (int64_t)o * 2 * h + i);
            acc = acc + w * x;
        }
        if (b_fc) acc = acc + load_elem(b_fc, is_bf16, o);
        fhat[o] = is_bf16 ? orc_bf16_to_f32(orc_f32_to_bf16(acc)) : acc;
    }
}

/* [notes04] §4.1-§4.2 and [zdszero] "draft 结构": the draft distribution comes from the
 * target's own frozen LM head, z = W_lm f^ (no bias, no norm in front of it).
 *   w_lm : [V][h] row-major;  z : [V] out.
 * Pin: float64 matrix product, within the fp32 dot-product bound. */
void orc_lm_head_row(int32_t h, int32_t V, int32_t is_bf16, const void *w_lm,
                     const float *fhat, float *z) {
#pragma omp parallel for schedule(static)
    for (int32_t v = 0; v < V; ++v) {
        float acc = 0.0f;
        for (int32_t i = 0; i < h; ++i)
            acc = acc + load_elem(w_lm, is_bf16, (int64_t)v * h + i) * fhat[i];
        z[v] = acc;
    }
}

/* True when (za, a) ranks strictly before (zb, b) in the order (value descending, index
 * ascending). */
static int ranks_before(float za, int32_t a, float zb, int32_t b) {
    return za > zb || (za == zb && a < b);
}

/* [notes04] §10.2 (the confidence of a drafted token is its draft probability) and §10.3
 * (each expanded node keeps its top-k children): per-row log-softmax and top-k.
 *   lse  = M + log(sum_v exp(z_v - M)),  M = max_v z_v   (sum in ascending v, fp32)
 *   ids  = the k best v by (z descending, v ascending)
 *   logp = z[ids] - lse
 * The j-th pick is the best element that ranks after pick j-1.
 * Pin: float64 logsumexp, and a full sort of the row by (-z, v). */
void orc_log_softmax_topk(int32_t V, int32_t k, const float *z, int32_t *ids, float *logp,
                          float *lse_out) {
    float M = z[0];
    for (int32_t v = 1; v < V; ++v)
        if (z[v] > M) M = z[v];
    float S = 0.0f;
    for (int32_t v = 0; v < V; ++v) S = S + expf(z[v] - M);
    float lse = M + logf(S);

    int32_t prev = -1;
    for (int32_t j = 0; j < k; ++j) {
        int32_t best = -1;
        for (int32_t v = 0; v < V; ++v) {
            if (prev >= 0 && !ranks_before(z[prev], prev, z[v], v)) continue; /* already taken */
            if (best < 0 || ranks_before(z[v], v, z[best], best)) best = v;
        }
        ids[j] = best;
        logp[j] = z[best] - lse;
        prev = best;
    }
    if (lse_out) *lse_out = lse;
}

/* Top-n of `count` scored items by (score descending, id ascending), where item i has id
 * ids[i].  Writes positions (0..count-1) into `out` in rank order.  Same pick-after-previous
 * rule as above. */
static void select_top(int32_t count, const float *score, const int32_t *ids, int32_t n,
                       int32_t *out) {
    int32_t prev = -1;
    for (int32_t j = 0; j < n; ++j) {
        int32_t best = -1;
        for (int32_t i = 0; i < count; ++i) {
            if (prev >= 0 && !ranks_before(score[prev], ids[prev], score[i], ids[i])) continue;
            if (best < 0 || ranks_before(score[i], ids[i], score[best], ids[best])) best = i;
        }
        out[j] = best;
        prev = best;
    }
}

/* ------------------------------------------------------------------------------------------ */
/* The draft-tree step                                                                        */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    int32_t batch;    /* B: independent requests */
    int32_t hidden;   /* h */
    int32_t vocab;    /* V */
    int32_t depth;    /* d: drafted levels = draft forwards ([zdszero] "在 SGLang 里": steps) */
    int32_t topk;     /* k: children per expanded node, frontier width */
    int32_t num_keep; /* m: drafted nodes kept by the rerank (the tree has m+1 with the root) */
    int32_t is_bf16;  /* weights, embedding and features are bf16 (else fp32) */
} orc_dims;

/* Candidates one request contributes to the rerank pool: the k children of the root, then
 * k*k for every further level ([zdszero] "在 SGLang 里": each level's top-k of k^2). */
int32_t orc_num_candidates(int32_t depth, int32_t k) { return k + (depth - 1) * k * k; }

/* Tree depth of candidate c (1 = child of the root).  Candidate ids are level-major:
 * 0..k-1 at depth 1, then k^2 per depth. */
static int32_t cand_depth(int32_t c, int32_t k) { return c < k ? 1 : 2 + (c - k) / (k * k); }

/*
 * One full draft-tree step for a batch of independent requests.
 *
 * Per request b ([notes04] §6.1 feature-level drafting, §10.3 expand + rerank; [zdszero]
 * "EAGLE-2" and "在 SGLang 里"; [jsqmd] "二、EAGLE-2" steps ① ②):
 *   level 0 : row x = [f_b || e(root_b)] -> f^ -> z -> top-k.  Its k children become
 *             candidates 0..k-1 with S = logp; the frontier is all k, in that order.
 *   level l : (l = 1..d-1) for frontier slot s (in frontier order) the row is
 *             x = [f^ of the row that produced the slot's node || e(token of that node)];
 *             child j becomes candidate k + (l-1)k^2 + s*k + j with
 *             S = fl(S_slot + logp_j); the next frontier (needed while l < d-1) is the top-k
 *             of these k^2 by (S desc, candidate asc).
 *   rerank  : the top-m of all candidates by (S desc, candidate asc).
 *   build   : tree index 0 is the root (position pos_base, parent -1, S = 0); the kept
 *             candidates in ascending candidate order take indices 1..m; parent = tree index
 *             of the parent candidate (0 for depth 1); position = depth + pos_base;
 *             mask bit j of row i is set iff j is i or an ancestor of i
 *             ([notes04] §12.5: ancestor-only mask, positions shared per level).
 *
 * Rows of level 0 are numbered b; rows of level l >= 1 are numbered b*k + s.
 * All per-row outputs are optional (NULL skips them); arrays are [depth][B*k][...], rows of
 * level 0 beyond B are left untouched.
 *   row_fhat [d][R][h], row_z [d][R][V], row_lse [d][R], row_ids/row_logp [d][R][k]
 *   front_cand [d][B][k] : candidate in each frontier slot entering level l (-1 at level 0)
 *   cand_tok/cand_S/cand_parent/cand_row [B][n_cand] : the rerank pool; cand_row is the row
 *             (within its producing level) whose f^ is the candidate's input feature
 *   tree_tok/tree_parent/tree_pos/tree_S/tree_cand [B][m+1], tree_mask [B][m+1][W],
 *             W = ceil((m+1)/32), bits packed LSB-first per 32-bit word
 *   node_z [B][m+1][V] : draft logits of every tree node's own row (the row that would expand
 *             it), used to synthesise target logits; optional.
 * Returns ORC_OK, ORC_ERR_ARG, ORC_ERR_TREE or ORC_ERR_NOMEM.
 */
int32_t orc_draft_tree(const orc_dims *dm, const void *w_fc, const void *b_fc, const void *w_lm,
                       const void *emb, const void *root_feat, const int32_t *root_tok,
                       const int32_t *pos_base, float *row_fhat, float *row_z, float *row_lse,
                       int32_t *row_ids, float *row_logp, int32_t *front_cand, int32_t *cand_tok,
                       float *cand_S, int32_t *cand_parent, int32_t *cand_row, int32_t *tree_tok,
                       int32_t *tree_parent, int32_t *tree_pos, uint32_t *tree_mask,
                       float *tree_S, int32_t *tree_cand, float *node_z) {
    const int32_t B = dm->batch, h = dm->hidden, V = dm->vocab, d = dm->depth, k = dm->topk;
    const int32_t m = dm->num_keep, bf = dm->is_bf16;
    if (B < 0 || h < 1 || V < 1 || d < 1 || k < 1 || k > V) return ORC_ERR_ARG;
    const int32_t n_cand = orc_num_candidates(d, k);
    if (m < 0 || m > n_cand) return ORC_ERR_ARG;
    if (!w_fc || !w_lm || !emb || !root_feat || !root_tok) return ORC_ERR_ARG;
    if (B == 0) return ORC_OK;

    const int64_t R = (int64_t)B * k;
    const int32_t n_nodes = m + 1;
    const int32_t W = (n_nodes + 31) / 32;

    /* scratch: f^ of every row of every level, one logit row, per-request pool and frontier */
    float *fh = (float *)malloc(sizeof(float) * (size_t)d * (size_t)R * (size_t)h);
    float *z = (float *)malloc(sizeof(float) * (size_t)V);
    float *feat = (float *)malloc(sizeof(float) * (size_t)h);
    float *x_fhat = (float *)malloc(sizeof(float) * (size_t)h);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    float *logp = (float *)malloc(sizeof(float) * (size_t)k);
    int32_t *p_tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_cand);
    float *p_S = (float *)malloc(sizeof(float) * (size_t)n_cand);
    int32_t *p_par = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_cand);
    int32_t *p_row = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_cand);
    int32_t *p_id = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_cand);
    int32_t *f_cand = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    float *f_S = (float *)malloc(sizeof(float) * (size_t)k);
    int32_t *pick = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_cand);
    int32_t *tree_of_cand = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_cand);
    int32_t *t_par = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_nodes);
    int32_t *t_cand = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_nodes);
    int32_t rc = ORC_OK;
    if (!fh || !z || !feat || !x_fhat || !ids || !logp || !p_tok || !p_S || !p_par || !p_row ||
        !p_id || !f_cand || !f_S || !pick || !tree_of_cand || !t_par || !t_cand) {
        rc = ORC_ERR_NOMEM;
        goto done;
    }

    for (int32_t b = 0; b < B; ++b) {
        /* ---------------- level 0: the root's row ---------------- */
        for (int32_t i = 0; i < h; ++i) feat[i] = load_elem(root_feat, bf, (int64_t)b * h + i);
        {
            const int64_t r = b;
            float *fo = fh + ((int64_t)0 * R + r) * h;
            orc_fc_row(h, bf, w_fc, b_fc, feat, emb, root_tok[b], fo);
            orc_lm_head_row(h, V, bf, w_lm, fo, z);
            float lse;
            orc_log_softmax_topk(V, k, z, ids, logp, &lse);
            if (row_fhat) memcpy(row_fhat + ((int64_t)0 * R + r) * h, fo, sizeof(float) * h);
            if (row_z) memcpy(row_z + ((int64_t)0 * R + r) * V, z, sizeof(float) * V);
            if (row_lse) row_lse[(int64_t)0 * R + r] = lse;
            if (row_ids) memcpy(row_ids + ((int64_t)0 * R + r) * k, ids, sizeof(int32_t) * k);
            if (row_logp) memcpy(row_logp + ((int64_t)0 * R + r) * k, logp, sizeof(float) * k);
            if (front_cand)
                for (int32_t s = 0; s < k; ++s) front_cand[((int64_t)0 * B + b) * k + s] = -1;
            for (int32_t j = 0; j < k; ++j) {
                p_tok[j] = ids[j];
                p_S[j] = logp[j];
                p_par[j] = -1;
                p_row[j] = (int32_t)r;
                f_cand[j] = j; /* the level-1 frontier is all k children, in child order */
                f_S[j] = logp[j];
            }
        }

        /* ---------------- levels 1..d-1: expand the frontier ---------------- */
        for (int32_t l = 1; l < d; ++l) {
            const int32_t base = k + (l - 1) * k * k;
            for (int32_t s = 0; s < k; ++s) {
                const int64_t r = (int64_t)b * k + s;
                const int32_t c_in = f_cand[s];
                const int32_t lvl_in = cand_depth(c_in, k) - 1; /* level whose row made c_in */
                const float *src = fh + ((int64_t)lvl_in * R + p_row[c_in]) * h;
                float *fo = fh + ((int64_t)l * R + r) * h;
                orc_fc_row(h, bf, w_fc, b_fc, src, emb, p_tok[c_in], fo);
                orc_lm_head_row(h, V, bf, w_lm, fo, z);
                float lse;
                orc_log_softmax_topk(V, k, z, ids, logp, &lse);
                if (row_fhat) memcpy(row_fhat + ((int64_t)l * R + r) * h, fo, sizeof(float) * h);
                if (row_z) memcpy(row_z + ((int64_t)l * R + r) * V, z, sizeof(float) * V);
                if (row_lse) row_lse[(int64_t)l * R + r] = lse;
                if (row_ids) memcpy(row_ids + ((int64_t)l * R + r) * k, ids, sizeof(int32_t) * k);
                if (row_logp)
                    memcpy(row_logp + ((int64_t)l * R + r) * k, logp, sizeof(float) * k);
                if (front_cand) front_cand[((int64_t)l * B + b) * k + s] = c_in;
                for (int32_t j = 0; j < k; ++j) {
                    const int32_t c = base + s * k + j;
                    p_tok[c] = ids[j];
                    p_S[c] = f_S[s] + logp[j];
                    p_par[c] = c_in;
                    p_row[c] = (int32_t)r;
                }
            }
            if (l < d - 1) {
                /* next frontier: top-k of this level's k^2 children by (S desc, cand asc) */
                for (int32_t i = 0; i < k * k; ++i) p_id[i] = base + i;
                select_top(k * k, p_S + base, p_id, k, pick);
                for (int32_t s = 0; s < k; ++s) {
                    f_cand[s] = base + pick[s];
                    f_S[s] = p_S[base + pick[s]];
                }
            }
        }

        /* ---------------- rerank: top-m of the whole pool ---------------- */
        for (int32_t c = 0; c < n_cand; ++c) {
            p_id[c] = c;
            tree_of_cand[c] = -1;
        }
        select_top(n_cand, p_S, p_id, m, pick);
        for (int32_t j = 0; j < m; ++j) tree_of_cand[pick[j]] = 1; /* mark kept */

        /* ---------------- build: level-major flattening ---------------- */
        t_par[0] = -1;
        t_cand[0] = -1;
        {
            int32_t t = 1;
            for (int32_t c = 0; c < n_cand; ++c)
                if (tree_of_cand[c] == 1) {
                    tree_of_cand[c] = t;
                    t_cand[t] = c;
                    ++t;
                }
        }
        for (int32_t t = 1; t < n_nodes; ++t) {
            const int32_t pc = p_par[t_cand[t]];
            if (pc < 0) {
                t_par[t] = 0;
            } else if (tree_of_cand[pc] >= 1) {
                t_par[t] = tree_of_cand[pc];
            } else {
                rc = ORC_ERR_TREE;
                goto done;
            }
        }
        for (int32_t t = 0; t < n_nodes; ++t) {
            const int64_t o = (int64_t)b * n_nodes + t;
            const int32_t c = t_cand[t];
            const int32_t dep = (t == 0) ? 0 : cand_depth(c, k);
            const int32_t pb = pos_base ? pos_base[b] : 0;
            if (tree_tok) tree_tok[o] = (t == 0) ? root_tok[b] : p_tok[c];
            if (tree_parent) tree_parent[o] = t_par[t];
            if (tree_pos) tree_pos[o] = dep + pb;
            if (tree_S) tree_S[o] = (t == 0) ? 0.0f : p_S[c];
            if (tree_cand) tree_cand[o] = c;
            if (tree_mask) {
                uint32_t *row = tree_mask + o * W;
                for (int32_t w = 0; w < W; ++w) row[w] = 0u;
                for (int32_t a = t; a >= 0; a = t_par[a]) row[a / 32] |= 1u << (a % 32);
            }
        }

        /* ---------------- draft logits of every tree node's own row ---------------- */
        if (node_z) {
            for (int32_t t = 0; t < n_nodes; ++t) {
                const float *src;
                int32_t tok;
                if (t == 0) {
                    for (int32_t i = 0; i < h; ++i)
                        feat[i] = load_elem(root_feat, bf, (int64_t)b * h + i);
                    src = feat;
                    tok = root_tok[b];
                } else {
                    const int32_t c = t_cand[t];
                    src = fh + ((int64_t)(cand_depth(c, k) - 1) * R + p_row[c]) * h;
                    tok = p_tok[c];
                }
                orc_fc_row(h, bf, w_fc, b_fc, src, emb, tok, x_fhat);
                orc_lm_head_row(h, V, bf, w_lm, x_fhat, node_z + ((int64_t)b * n_nodes + t) * V);
            }
        }

        /* ---------------- pool out ---------------- */
        for (int32_t c = 0; c < n_cand; ++c) {
            const int64_t o = (int64_t)b * n_cand + c;
            if (cand_tok) cand_tok[o] = p_tok[c];
            if (cand_S) cand_S[o] = p_S[c];
            if (cand_parent) cand_parent[o] = p_par[c];
            if (cand_row) cand_row[o] = p_row[c];
        }
    }

done:
    free(fh); free(z); free(feat); free(x_fhat); free(ids); free(logp);
    free(p_tok); free(p_S); free(p_par); free(p_row); free(p_id); free(f_cand); free(f_S);
    free(pick); free(tree_of_cand); free(t_par); free(t_cand);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* Draft decoder layer with tree attention over a draft KV cache                              */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    int32_t batch;     /* B */
    int32_t nodes;     /* n: tree nodes (root first, parents before children) */
    int32_t prefix;    /* P: cached positions before the tree */
    int32_t hidden;    /* h */
    int32_t heads;     /* H query heads */
    int32_t kv_heads;  /* Hkv, divides H */
    int32_t head_dim;  /* D, even */
    int32_t inter;     /* I: MLP width */
    float rope_theta;  /* RoPE base */
    float rms_eps;     /* RMSNorm epsilon */
} orc_layer_dims;

static float bf16r(float x) { return orc_bf16_to_f32(orc_f32_to_bf16(x)); }

/* y[o] = sum_i W[o][i] x[i], fp32, ascending i; W bf16 [out][in]. */
static void orc_matvec_bf16(const uint16_t *W, int32_t out, int32_t in, const float *x, float *y) {
#pragma omp parallel for schedule(static)
    for (int32_t o = 0; o < out; ++o) {
        float acc = 0.0f;
        for (int32_t i = 0; i < in; ++i) acc = acc + orc_bf16_to_f32(W[(int64_t)o * in + i]) * x[i];
        y[o] = acc;
    }
}

/* Llama's rotary embedding ("rotate half"): for j < D/2, angle = pos * theta^(-2j/D), and the
 * pair (x[j], x[j + D/2]) is rotated by it.  Angles, sines and cosines in double precision. */
static void orc_rope(float *x, int32_t D, int32_t pos, double theta) {
    const int32_t half = D / 2;
    for (int32_t j = 0; j < half; ++j) {
        const double ang = (double)pos * pow(theta, -2.0 * j / (double)D);
        const double c = cos(ang), sn = sin(ang);
        const double a = x[j], b = x[j + half];
        x[j] = (float)(a * c - b * sn);
        x[j + half] = (float)(b * c + a * sn);
    }
}

/*
 * [zdszero] "在 SGLang 里" (the draft model: embedding, fc = Linear(2h, h, bias), one Llama decoder
 * layer whose first input_layernorm is the identity, no final norm, the target's lm_head) and
 * [notes04] §4.1 (FC, then a light decoder layer predicts the next feature) and §12.5 (tree
 * attention: each node sees its ancestors only; positions shared per depth).  One decoder layer over
 * the n nodes of each request's tree; each node attends to the P cached positions (keys stored
 * already rotated) and to the tree nodes its mask row marks (itself and its ancestors).  Rounding
 * points (a bf16 model): each projection's output, the attention output, each residual sum, the
 * normed activation and the MLP product are rounded to bf16; dot products, softmax and norms are fp32.
 *   x_i   -> qkv = Wqkv x_i (rows: H*D q, Hkv*D k, Hkv*D v), q and k rotated at pos[i]
 *   attn  -> for head hq (kv head hq / (H / Hkv)): s_j = q.k_j / sqrt(D) over visible keys,
 *            p = softmax(s), o = sum p_j v_j
 *   h1    =  x_i + Wo o
 *   r     =  RMSNorm(h1) * w_norm      (post-attention norm; the input norm is the identity)
 *   a     =  silu(g) * u,  [g; u] = Wgu r
 *   out_i =  h1 + Wd a
 * Inputs (bf16 as uint16): x [B][n][h], Wqkv [(H+2Hkv)D][h], Wo [h][H D], w_norm [h], Wgu [2I][h],
 * Wd [h][I], k_cache / v_cache [B][P][Hkv][D], pos [B][n], mask [B][n][W] (bit t of row i: node t
 * visible to node i).  Outputs: out [B][n][h] (bf16 bits), and optionally the tree's rotated keys
 * and values k_new / v_new [B][n][Hkv][D] (bf16 bits), which extend the cache.
 * Pins: attention over a chain with no prefix against float64 causal attention; RoPE's relative
 * position property; the whole layer against a float64 restatement within bf16 tolerances.
 */
int32_t orc_decoder_layer(const orc_layer_dims *L, const uint16_t *x, const uint16_t *Wqkv,
                          const uint16_t *Wo, const uint16_t *w_norm, const uint16_t *Wgu,
                          const uint16_t *Wd, const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *pos, const uint32_t *mask, uint16_t *out,
                          uint16_t *k_new, uint16_t *v_new) {
    const int32_t B = L->batch, n = L->nodes, P = L->prefix, h = L->hidden, H = L->heads;
    const int32_t Hk = L->kv_heads, D = L->head_dim, I = L->inter, W = (n + 31) / 32;
    if (B < 0 || n < 1 || P < 0 || h < 1 || H < 1 || Hk < 1 || H % Hk || D < 2 || D % 2 || I < 1)
        return ORC_ERR_ARG;
    const int32_t nq = H * D, nk = Hk * D, nqkv = nq + 2 * nk, grp = H / Hk;
    float *xin = (float *)malloc(sizeof(float) * (size_t)h);
    float *qkv = (float *)malloc(sizeof(float) * (size_t)n * nqkv);  /* one request's tree */
    float *o = (float *)malloc(sizeof(float) * (size_t)nq);
    float *t = (float *)malloc(sizeof(float) * (size_t)(h > 2 * I ? h : 2 * I));
    float *h1 = (float *)malloc(sizeof(float) * (size_t)h);
    float *r = (float *)malloc(sizeof(float) * (size_t)h);
    float *a = (float *)malloc(sizeof(float) * (size_t)I);
    float *sc = (float *)malloc(sizeof(float) * (size_t)(P + n));
    int32_t rc = ORC_OK;
    if (!xin || !qkv || !o || !t || !h1 || !r || !a || !sc) {
        rc = ORC_ERR_NOMEM;
        goto done;
    }
    const float inv_sqrt_d = 1.0f / sqrtf((float)D);
    for (int32_t b = 0; b < B; ++b) {
        /* projections and rotations of every node of this tree */
        for (int32_t i = 0; i < n; ++i) {
            const uint16_t *xr = x + ((int64_t)b * n + i) * h;
            for (int32_t e = 0; e < h; ++e) xin[e] = orc_bf16_to_f32(xr[e]);
            float *q = qkv + (int64_t)i * nqkv;
            orc_matvec_bf16(Wqkv, nqkv, h, xin, q);
            for (int32_t e = 0; e < nqkv; ++e) q[e] = bf16r(q[e]);
            const int32_t p = pos[(int64_t)b * n + i];
            for (int32_t hh = 0; hh < H; ++hh) orc_rope(q + hh * D, D, p, L->rope_theta);
            for (int32_t hh = 0; hh < Hk; ++hh) orc_rope(q + nq + hh * D, D, p, L->rope_theta);
            for (int32_t e = 0; e < nq + nk; ++e) q[e] = bf16r(q[e]);
            if (k_new && v_new)
                for (int32_t e = 0; e < nk; ++e) {
                    k_new[((int64_t)b * n + i) * nk + e] = orc_f32_to_bf16(q[nq + e]);
                    v_new[((int64_t)b * n + i) * nk + e] = orc_f32_to_bf16(q[nq + nk + e]);
                }
        }
        for (int32_t i = 0; i < n; ++i) {
            const float *q = qkv + (int64_t)i * nqkv;
            const uint32_t *mrow = mask + ((int64_t)b * n + i) * W;
            for (int32_t hq = 0; hq < H; ++hq) {
                const int32_t hk = hq / grp;
                /* scores over the visible keys: the cache, then the marked tree nodes */
                float mx = -HUGE_VALF;
                int32_t cnt = 0;
                for (int32_t j = 0; j < P; ++j) {
                    const uint16_t *kr = k_cache + (((int64_t)b * P + j) * Hk + hk) * D;
                    float s = 0.0f;
                    for (int32_t e = 0; e < D; ++e) s = s + q[hq * D + e] * orc_bf16_to_f32(kr[e]);
                    sc[cnt++] = s * inv_sqrt_d;
                }
                for (int32_t tn = 0; tn < n; ++tn) {
                    if (!((mrow[tn / 32] >> (tn % 32)) & 1u)) continue;
                    const float *kr = qkv + (int64_t)tn * nqkv + nq + hk * D;
                    float s = 0.0f;
                    for (int32_t e = 0; e < D; ++e) s = s + q[hq * D + e] * kr[e];
                    sc[cnt++] = s * inv_sqrt_d;
                }
                for (int32_t j = 0; j < cnt; ++j)
                    if (sc[j] > mx) mx = sc[j];
                float den = 0.0f;
                for (int32_t j = 0; j < cnt; ++j) {
                    sc[j] = expf(sc[j] - mx);
                    den = den + sc[j];
                }
                for (int32_t e = 0; e < D; ++e) {
                    float acc = 0.0f;
                    int32_t c = 0;
                    for (int32_t j = 0; j < P; ++j, ++c)
                        acc = acc + sc[c] * orc_bf16_to_f32(v_cache[(((int64_t)b * P + j) * Hk + hk) * D + e]);
                    for (int32_t tn = 0; tn < n; ++tn) {
                        if (!((mrow[tn / 32] >> (tn % 32)) & 1u)) continue;
                        acc = acc + sc[c++] * qkv[(int64_t)tn * nqkv + nq + nk + hk * D + e];
                    }
                    o[hq * D + e] = bf16r(acc / den);
                }
            }
            /* output projection and residual */
            const uint16_t *xr = x + ((int64_t)b * n + i) * h;
            orc_matvec_bf16(Wo, h, nq, o, t);
            for (int32_t e = 0; e < h; ++e) h1[e] = bf16r(orc_bf16_to_f32(xr[e]) + t[e]);
            /* post-attention RMSNorm */
            float ss = 0.0f;
            for (int32_t e = 0; e < h; ++e) ss = ss + h1[e] * h1[e];
            const float inv = 1.0f / sqrtf(ss / (float)h + L->rms_eps);
            for (int32_t e = 0; e < h; ++e) r[e] = bf16r(h1[e] * inv * orc_bf16_to_f32(w_norm[e]));
            /* SwiGLU MLP and residual */
            orc_matvec_bf16(Wgu, 2 * I, h, r, t);
            for (int32_t e = 0; e < I; ++e) {
                const float g = bf16r(t[e]), u = bf16r(t[I + e]);
                a[e] = bf16r(g / (1.0f + expf(-g)) * u);
            }
            orc_matvec_bf16(Wd, h, I, a, t);
            uint16_t *orow = out + ((int64_t)b * n + i) * h;
            for (int32_t e = 0; e < h; ++e) orow[e] = orc_f32_to_bf16(h1[e] + t[e]);
        }
    }
done:
    free(xin); free(qkv); free(o); free(t); free(h1); free(r); free(a); free(sc);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* EAGLE-1 static tree                                                                         */
/* ------------------------------------------------------------------------------------------ */

/*
 * [notes04] §10.1 and §12 item 7: EAGLE-1 (like Medusa) drafts a tree of fixed shape, the same
 * for every context - its shape is set by position only; [zdszero] "EAGLE：特征级自回归 + 前移一位
 * 的 token": inference uses one static draft tree, verified with the ancestor-only mask.  The
 * pages give no format for the shape; the reading here: drafted node j (1..N) is given as
 * (parent p_j, rank r_j): the r_j-th most probable token (0-based, ties to the lower id) of the
 * draft distribution at its parent.  Nodes are listed with parents first and depth
 * non-decreasing; siblings carry distinct ranks.
 * For request b: node 0 is the root (root feature, root token).  For every node j that has a child,
 * its row [feat_in(j) || E[tok_j]] goes through FC -> LM head -> log-softmax + top-K_j (K_j = the
 * largest rank among its children + 1); child c takes tok_c = ids[r_c], S_c = fl(S_j + logp[r_c])
 * and feat_in(c) = f^_j (feat_in(root) = the root feature, S_root = 0).
 * Outputs [B][N+1]: tree_tok, tree_parent (-1 for the root), tree_pos (depth + pos_base),
 * tree_mask [B][N+1][W] (ancestor-only, LSB first), tree_S.  node_fhat [B][N+1][h] (f^ of the
 * rows of nodes with children; zero elsewhere) optional.
 * Pins: a rank-0 chain equals the dynamic tree with topk = 1; a depth-1 star of the top k equals
 * the dynamic tree with depth 1 and m = k; a full binary tree against its construction in the
 * test from the row functions.
 */
int32_t orc_draft_static(const orc_dims *dm, const void *w_fc, const void *b_fc, const void *w_lm,
                         const void *emb, const void *root_feat, const int32_t *root_tok,
                         const int32_t *pos_base, int32_t n_static, const int32_t *spec,
                         int32_t *tree_tok, int32_t *tree_parent, int32_t *tree_pos,
                         uint32_t *tree_mask, float *tree_S, float *node_fhat) {
    const int32_t B = dm->batch, h = dm->hidden, V = dm->vocab, bf = dm->is_bf16;
    const int32_t n = n_static + 1, W = (n + 31) / 32;
    if (B < 0 || h < 1 || V < 1 || n_static < 0 || !spec) return ORC_ERR_ARG;
    int32_t *dep = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t *kmax = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    float *fh = (float *)malloc(sizeof(float) * (size_t)n * (size_t)h);
    float *feat = (float *)malloc(sizeof(float) * (size_t)h);
    float *z = (float *)malloc(sizeof(float) * (size_t)V);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * 16);
    float *logp = (float *)malloc(sizeof(float) * 16);
    int32_t rc = ORC_OK;
    if (!dep || !kmax || !fh || !feat || !z || !ids || !logp) {
        rc = ORC_ERR_NOMEM;
        goto done;
    }
    /* the shape: depths, and each node's number of top-k entries its children need */
    dep[0] = 0;
    for (int32_t j = 0; j < n; ++j) kmax[j] = 0;
    for (int32_t j = 1; j < n; ++j) {
        const int32_t p = spec[2 * (j - 1)], r = spec[2 * (j - 1) + 1];
        if (p < 0 || p >= j || r < 0 || r >= 16 || r >= V) {
            rc = ORC_ERR_ARG;
            goto done;
        }
        dep[j] = dep[p] + 1;
        if (dep[j] < dep[j - 1]) { /* depth must not decrease */
            rc = ORC_ERR_ARG;
            goto done;
        }
        for (int32_t i = 1; i < j; ++i)
            if (spec[2 * (i - 1)] == p && spec[2 * (i - 1) + 1] == r) { /* sibling with the same rank */
                rc = ORC_ERR_ARG;
                goto done;
            }
        if (r + 1 > kmax[p]) kmax[p] = r + 1;
    }
    for (int32_t b = 0; b < B; ++b) {
        int32_t *tt = tree_tok + (int64_t)b * n;
        int32_t *tp = tree_parent + (int64_t)b * n;
        float *tS = tree_S + (int64_t)b * n;
        const int32_t pb = pos_base ? pos_base[b] : 0;
        tt[0] = root_tok[b];
        tp[0] = -1;
        tS[0] = 0.0f;
        for (int32_t j = 1; j < n; ++j) tp[j] = spec[2 * (j - 1)];
        /* nodes in order: a node's row is evaluated before any of its children is read */
        for (int32_t j = 0; j < n; ++j) {
            /* tt[j] and tS[j] were set when its parent's row was evaluated */
            if (kmax[j] == 0) continue;
            const float *in;
            if (j == 0) {
                for (int32_t i = 0; i < h; ++i) feat[i] = load_elem(root_feat, bf, (int64_t)b * h + i);
                in = feat;
            } else {
                in = fh + (int64_t)tp[j] * h;
            }
            if (tt[j] < 0 || tt[j] >= V) {
                rc = ORC_ERR_ARG;
                goto done;
            }
            orc_fc_row(h, bf, w_fc, b_fc, in, emb, tt[j], fh + (int64_t)j * h);
            orc_lm_head_row(h, V, bf, w_lm, fh + (int64_t)j * h, z);
            float lse;
            orc_log_softmax_topk(V, kmax[j], z, ids, logp, &lse);
            for (int32_t c = j + 1; c < n; ++c) {
                if (spec[2 * (c - 1)] != j) continue;
                const int32_t r = spec[2 * (c - 1) + 1];
                tt[c] = ids[r];
                tS[c] = tS[j] + logp[r];
            }
        }
        for (int32_t j = 0; j < n; ++j) {
            tree_pos[(int64_t)b * n + j] = dep[j] + pb;
            uint32_t *mrow = tree_mask + ((int64_t)b * n + j) * W;
            for (int32_t w = 0; w < W; ++w) mrow[w] = 0u;
            for (int32_t x = j; x >= 0; x = tp[x]) mrow[x / 32] |= 1u << (x % 32);
            if (node_fhat) {
                float *o = node_fhat + ((int64_t)b * n + j) * h;
                for (int32_t i = 0; i < h; ++i) o[i] = kmax[j] ? fh[(int64_t)j * h + i] : 0.0f;
            }
        }
    }
done:
    free(dep); free(kmax); free(fh); free(feat); free(z); free(ids); free(logp);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* Draft extend: the next round's root                                                        */
/* ------------------------------------------------------------------------------------------ */

/*
 * [zdszero] "在 SGLang 里": one decode step is one target verify, (steps - 1) draft forwards and
 * one draft extend; the draft's own features along the tree are guesses, so after the verify the
 * draft runs again over the verified positions with the target's true hidden states and the
 * accepted tokens, and the last verified position is where the next round starts (its top-k is
 * the next round's first level).  [notes04] §6.2 and §12 item 3: the true features of the
 * accepted path start the next round's draft.
 * For request b, with path nodes a_0 = 0 (the root), a_1 .. a_L (L = accept_len[b]) and the
 * tokens that follow them accept_tok[b][0..L] (the accepted tokens, then the bonus):
 *   row i (0 <= i <= L) = [F[b][a_i] || E[accept_tok[b][i]]]
 *   f^_i = FC(row i) (rounded once to bf16 for bf16), z_i = LM_head(f^_i)
 *   next root: feature F[b][a_L], token accept_tok[b][L]; its level-0 row is row L, whose
 *   log-softmax and top-k are returned (the next round's first level).
 * Rows L < i <= depth of the [B][depth+1] outputs repeat row L.
 *   node_feat [B][n_nodes][h] fp32 (bf16 features widened exactly), outputs: next_feat [B][h],
 *   next_tok [B], path_fhat [B][depth+1][h], path_z [B][depth+1][V] (or NULL), ids / logp [B][k],
 *   lse [B].
 * Pins: row L equals orc_draft_tree's level-0 row for the root (F[b][a_L], bonus); the path rows
 * against their construction by hand in the test.
 */
int32_t orc_draft_extend(const orc_dims *dm, const void *w_fc, const void *b_fc, const void *w_lm,
                         const void *emb, const float *node_feat, int32_t n_nodes,
                         const int32_t *accept_len, const int32_t *accept_nodes,
                         const int32_t *accept_tok, float *next_feat, int32_t *next_tok,
                         float *path_fhat, float *path_z, int32_t *ids, float *logp, float *lse) {
    const int32_t B = dm->batch, h = dm->hidden, V = dm->vocab, d = dm->depth, k = dm->topk;
    const int32_t bf = dm->is_bf16;
    if (B < 0 || h < 1 || V < 1 || d < 1 || k < 1 || k > V || n_nodes < 1) return ORC_ERR_ARG;
    float *z = (float *)malloc(sizeof(float) * (size_t)V);
    float *fo = (float *)malloc(sizeof(float) * (size_t)h);
    if (!z || !fo) {
        free(z); free(fo);
        return ORC_ERR_NOMEM;
    }
    for (int32_t b = 0; b < B; ++b) {
        const int32_t L = accept_len[b];
        if (L < 0 || L > d) {
            free(z); free(fo);
            return ORC_ERR_ARG;
        }
        for (int32_t i = 0; i <= d; ++i) {
            const int32_t r = i <= L ? i : L;
            const int32_t node = accept_nodes[(int64_t)b * (d + 1) + r];
            const int32_t tok = accept_tok[(int64_t)b * (d + 1) + r];
            if (node < 0 || node >= n_nodes || tok < 0 || tok >= V) {
                free(z); free(fo);
                return ORC_ERR_ARG;
            }
            const float *feat = node_feat + ((int64_t)b * n_nodes + node) * h;
            orc_fc_row(h, bf, w_fc, b_fc, feat, emb, tok, fo);
            orc_lm_head_row(h, V, bf, w_lm, fo, z);
            memcpy(path_fhat + ((int64_t)b * (d + 1) + i) * h, fo, sizeof(float) * (size_t)h);
            if (path_z) memcpy(path_z + ((int64_t)b * (d + 1) + i) * V, z, sizeof(float) * (size_t)V);
            if (i == L) {
                orc_log_softmax_topk(V, k, z, ids + (int64_t)b * k, logp + (int64_t)b * k, lse + b);
                memcpy(next_feat + (int64_t)b * h, feat, sizeof(float) * (size_t)h);
                next_tok[b] = tok;
            }
        }
    }
    free(z);
    free(fo);
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Greedy tree verification                                                                   */
/* ------------------------------------------------------------------------------------------ */

/*
 * [notes04] §6.2 (the target scores every tree node in one forward, verification walks the
 * tree from the root), [zdszero] "Medusa" (at temperature 0 acceptance reduces to greedy) and
 * [jsqmd] "二、EAGLE-2" (accept the longest consistent root path, then continue from its last
 * node).  For request b:
 *   g_i  = argmax_v T[b][i][v], ties to the lowest v
 *   walk : cur = 0 (root); while some child c of cur has token(c) == g_cur: accept c, cur = c
 *          (siblings carry distinct tokens, so at most one child matches; the lowest index is
 *          taken if an input breaks that)
 *   out  : accept_len = number of drafted nodes accepted (0..depth);
 *          accept_nodes[0..accept_len] = the path's tree indices, root first;
 *          accept_tok[0..accept_len-1] = their tokens, accept_tok[accept_len] = g_cur (the
 *          bonus token); unused slots -1.  Both outputs are [B][depth+1].
 * T is [B][n_nodes][V] fp32.  g_out [B][n_nodes] is optional.
 * Pins: brute force over every root path of small random trees; the expected committed
 * tokens per round against the worked values of [notes04] §8 and exercise 2.
 */
int32_t orc_verify_greedy(int32_t B, int32_t n_nodes, int32_t V, int32_t depth,
                          const int32_t *tree_tok, const int32_t *tree_parent, const float *T,
                          int32_t *g_out, int32_t *accept_len, int32_t *accept_nodes,
                          int32_t *accept_tok) {
    if (B < 0 || n_nodes < 1 || V < 1 || depth < 0) return ORC_ERR_ARG;
    int32_t *g = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_nodes > 0 ? n_nodes : 1));
    if (!g) return ORC_ERR_NOMEM;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t *tok = tree_tok + (int64_t)b * n_nodes;
        const int32_t *par = tree_parent + (int64_t)b * n_nodes;
        for (int32_t i = 0; i < n_nodes; ++i) {
            const float *row = T + ((int64_t)b * n_nodes + i) * V;
            int32_t best = 0;
            for (int32_t v = 1; v < V; ++v)
                if (row[v] > row[best]) best = v;
            g[i] = best;
            if (g_out) g_out[(int64_t)b * n_nodes + i] = best;
        }
        int32_t *an = accept_nodes + (int64_t)b * (depth + 1);
        int32_t *at = accept_tok + (int64_t)b * (depth + 1);
        for (int32_t i = 0; i <= depth; ++i) {
            an[i] = -1;
            at[i] = -1;
        }
        int32_t cur = 0, n = 0;
        an[0] = 0;
        while (n < depth) {
            int32_t next = -1;
            for (int32_t c = 1; c < n_nodes; ++c)
                if (par[c] == cur && tok[c] == g[cur]) {
                    next = c;
                    break;
                }
            if (next < 0) break;
            at[n] = tok[next];
            ++n;
            an[n] = next;
            cur = next;
        }
        at[n] = g[cur];
        accept_len[b] = n;
    }
    free(g);
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Sampling tree verification (recursive rejection sampling; threshold variant)               */
/* ------------------------------------------------------------------------------------------ */

/*
 * [notes04] §6.2 "验证阶段（树注意力 + 递归拒绝采样）": the target scores every tree node in one
 * forward; then, node by node from the root, a drafted token t is accepted when a uniform r
 * satisfies r <= min(1, p(t) / q(t)), and on rejection the distribution to draw from becomes
 * norm(max(0, p - q)); with several drafted children the same step is repeated child after
 * child on the updated p (the multi-candidate form of SpecInfer, which [notes04] names as the
 * framework of EAGLE's tree verification).  [notes04] §7.1: with q == p every test passes.
 * [tomjerr] "Summary" (the SGLang note): the threshold variant accepts a drafted token when its
 * target probability passes a threshold and draws the bonus token by one rejection step over
 * the layer only when every child fails.
 *
 * Readings where the pages leave a step open (each is listed in the design notes):
 *   - p_i = softmax(T[b][i] / temperature) and q_i = softmax(Z[b][i] / temperature): T and Z are
 *     the target's and the draft's logits at node i, i.e. the distributions of the token that
 *     follows node i (q_i is what node i's children were drafted from); temperature > 0;
 *   - children of a node are visited in ascending tree index (the draft's own ranking, since the
 *     tree lists a parent's kept children by candidate id);
 *   - the test of child c uses its own uniform u_acc[b][c]: accept iff P(t_c) > 0 and
 *     u_acc * q(t_c) <= P(t_c) (the division-free form of u <= min(1, P/q); a token the target
 *     gives probability 0 is never accepted);
 *   - after a rejection P <- max(0, P - q) / sum; if that sum is 0 (P == q up to rounding),
 *     P is left as it was;
 *   - threshold mode (mode 1): the first child c with p_cur(t_c) >= threshold is accepted; if
 *     none is, P = p_cur updated by one rejection step per child in order, and the bonus is drawn
 *     from it;
 *   - the bonus token is drawn from the final P by inverse CDF with u_bonus[b]: the smallest v
 *     whose running sum (ascending v) exceeds u_bonus * sum(P); if rounding leaves none, the
 *     largest v with P(v) > 0.
 * Everything is computed in double precision.
 * Outputs as in orc_verify_greedy: accept_len [B], accept_nodes / accept_tok [B][depth+1]
 * (bonus last, unused slots -1).
 * Pins: worked examples derived by hand (tests/golden/verify_sample_cases.json); with q == p the
 * first child is always accepted ([notes04] §7.1); losslessness: with children drawn from q the
 * first emitted token is distributed as p (chi-square over many draws); greedy limit of the
 * threshold mode.
 */
static void orc_softmax_scaled(const float *logits, int32_t V, double inv_temp, double *out) {
    double m = -HUGE_VAL;
    for (int32_t v = 0; v < V; ++v)
        if ((double)logits[v] * inv_temp > m) m = (double)logits[v] * inv_temp;
    double s = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        out[v] = exp((double)logits[v] * inv_temp - m);
        s += out[v];
    }
    for (int32_t v = 0; v < V; ++v) out[v] /= s;
}

/* P <- norm(max(0, P - q)); P is left unchanged when the residual is empty. */
static void orc_residual(double *P, const double *q, int32_t V) {
    double s = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        const double r = P[v] - q[v];
        s += r > 0.0 ? r : 0.0;
    }
    if (!(s > 0.0)) return;
    for (int32_t v = 0; v < V; ++v) {
        const double r = P[v] - q[v];
        P[v] = (r > 0.0 ? r : 0.0) / s;
    }
}

static int32_t orc_inverse_cdf(const double *P, int32_t V, double u) {
    double tot = 0.0;
    for (int32_t v = 0; v < V; ++v) tot += P[v];
    const double target = u * tot;
    double run = 0.0;
    int32_t last = -1;
    for (int32_t v = 0; v < V; ++v) {
        if (P[v] > 0.0) last = v;
        run += P[v];
        if (run > target && P[v] > 0.0) return v;
    }
    return last < 0 ? 0 : last;
}

int32_t orc_verify_sample(int32_t B, int32_t n_nodes, int32_t V, int32_t depth,
                          const int32_t *tree_tok, const int32_t *tree_parent, const float *T,
                          const float *Z, double temperature, int32_t mode, double threshold,
                          const float *u_acc, const float *u_bonus, int32_t *accept_len,
                          int32_t *accept_nodes, int32_t *accept_tok) {
    if (B < 0 || n_nodes < 1 || V < 1 || depth < 0 || !(temperature > 0.0) || mode < 0 || mode > 1)
        return ORC_ERR_ARG;
    double *P = (double *)malloc(sizeof(double) * (size_t)V);
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    if (!P || !q) {
        free(P); free(q);
        return ORC_ERR_NOMEM;
    }
    const double inv_t = 1.0 / temperature;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t *tok = tree_tok + (int64_t)b * n_nodes;
        const int32_t *par = tree_parent + (int64_t)b * n_nodes;
        int32_t *an = accept_nodes + (int64_t)b * (depth + 1);
        int32_t *at = accept_tok + (int64_t)b * (depth + 1);
        for (int32_t i = 0; i <= depth; ++i) {
            an[i] = -1;
            at[i] = -1;
        }
        int32_t cur = 0, n = 0;
        an[0] = 0;
        for (;;) {
            const float *trow = T + ((int64_t)b * n_nodes + cur) * V;
            const float *zrow = Z + ((int64_t)b * n_nodes + cur) * V;
            orc_softmax_scaled(trow, V, inv_t, P); /* p_cur */
            orc_softmax_scaled(zrow, V, inv_t, q); /* q_cur */
            int32_t next = -1;
            if (n < depth) {
                if (mode == 0) {
                    for (int32_t c = 1; c < n_nodes && next < 0; ++c) {
                        if (par[c] != cur) continue;
                        const int32_t t = tok[c];
                        const double u = (double)u_acc[(int64_t)b * n_nodes + c];
                        if (P[t] > 0.0 && u * q[t] <= P[t]) next = c;
                        else orc_residual(P, q, V);
                    }
                } else {
                    for (int32_t c = 1; c < n_nodes && next < 0; ++c)
                        if (par[c] == cur && P[tok[c]] >= threshold) next = c;
                    if (next < 0)
                        for (int32_t c = 1; c < n_nodes; ++c)
                            if (par[c] == cur) orc_residual(P, q, V);
                }
            }
            if (next < 0) break;
            at[n] = tok[next];
            ++n;
            an[n] = next;
            cur = next;
        }
        at[n] = orc_inverse_cdf(P, V, (double)u_bonus[b]);
        accept_len[b] = n;
    }
    free(P);
    free(q);
    return ORC_OK;
}

/* Element-wise bf16 rounding of an fp32 array (test helper for the rounding pin). */
void orc_round_bf16_array(int64_t n, const float *in, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}
