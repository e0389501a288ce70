/*
 * eagle_tree.h - C ABI of the GB300 (sm_103a) EAGLE / EAGLE-2 dynamic draft-tree engine.
 *
 * One draft-tree step, as the pages describe it:
 *   draft level l = 0..d-1   for every frontier node, concatenate the feature with the embedding
 *                            of the node's (shifted) token, apply the draft FC (2h -> h, bias) and
 *                            the target's frozen LM head (h -> V), take the log-softmax and the
 *                            top-k children, and expand: a child's path score is its parent's
 *                            plus its own log-probability, and the top-k of the k*k children
 *                            become the next frontier;
 *   rerank + build           keep the top-m drafted nodes of the whole pool and flatten them into
 *                            a tree: parent indices, depth positions, ancestor-only mask;
 *   verify                   greedy: the longest root path whose every node is the target's
 *                            argmax at its parent, plus the bonus token.
 * Sources (web pages, by title and section):
 *   "EAGLE 推测解码为什么比 Medusa 快？（含 EAGLE-2 动态草稿树）" (zzszmyf notes ch. 04): §4.1 the
 *       draft model [f || e(t)] -> FC -> shared LM head; §6.1 feature-level drafting; §6.2 tree
 *       verification; §10.2 confidence; §10.3 expand + rerank and its two properties; §12.5
 *       ancestor-only mask, positions shared per level.
 *   zdszero Medusa -> EAGLE -> EAGLE-2 notes: "draft 结构" (fc = Linear(2h, h, bias=True)),
 *       "EAGLE-2" (expand: top-k per level; rerank: top-m of all drafted tokens), "在 SGLang 里"
 *       (steps / topk / num_draft_tokens = depth / k / m + 1, and the per-level top-k of k^2).
 *   "投机解码：从eagle1到dflash" (jsqmd), "二、EAGLE-2": flatten, positions, tree mask, accept the
 *       longest consistent root path.
 *
 * Conventions shared by every entry point:
 *   - All device memory is owned by the caller.  The library allocates no device memory: the
 *     handle works inside a caller-provided workspace, and weights are borrowed (they must
 *     outlive the handle).  Only host-side objects are allocated: the handle, by eagle_tree_init,
 *     and the pinned staging, side stream and events of eagle_tree_step_host, by its first call.
 *   - Every call that takes a stream only enqueues work on it: no host synchronisation, no
 *     allocation.  The exceptions are eagle_tree_init (which clears its workspace with a
 *     synchronous cudaMemset), eagle_tree_status and eagle_tree_step_host (which synchronise
 *     the stream they are given).
 *   - Argument and shape errors are detected on the host and returned before anything is
 *     launched.  Errors detected inside a kernel (a bounded wait that ran out, an index out of
 *     range, a rerank that broke the tree property) are latched in a device status word that
 *     eagle_tree_status reads and clears.
 *   - A handle serves one stream at a time; calls on one handle must be ordered on one stream.
 *   - Integer arrays are int32, row-major, C order.  "bf16" is IEEE-754 binary32 truncated to
 *     its upper 16 bits (round to nearest even when produced).
 *   - Device pointers must be 16-byte aligned; the workspace 256-byte aligned.
 */
#ifndef EAGLE_TREE_H
#define EAGLE_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define EAGLE_API __attribute__((visibility("default")))
#else
#define EAGLE_API
#endif

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st *eagle_stream_t;

typedef enum {
    EAGLE_OK = 0,
    EAGLE_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned pointer, short workspace */
    EAGLE_ERR_UNSUPPORTED = 2,    /* valid request outside what this build handles */
    EAGLE_ERR_STATE = 3,          /* calls out of order (levels 0..d-1, then rerank) */
    EAGLE_ERR_CUDA = 4,           /* a CUDA runtime call failed */
    EAGLE_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait ran out (read by eagle_tree_status) */
    EAGLE_ERR_DEVICE_BOUNDS = 6   /* a kernel saw an out-of-range index or a broken tree */
} eagle_status;

typedef enum { EAGLE_F32 = 0, EAGLE_BF16 = 1 } eagle_dtype;

/*
 * The engine's configuration.  Knob names follow the SGLang flags quoted on the zdszero page
 * ("在 SGLang 里"): depth = --speculative-num-steps, topk = --speculative-eagle-topk,
 * num_keep + 1 = --speculative-num-draft-tokens (the tree counts the root).
 *   batch     B >= 0 independent requests (0: every call is a no-op)
 *   hidden    h >= 1 (a multiple of 8 for bf16, of 4 for fp32)
 *   vocab     V >= topk
 *   depth     d in [1, 32]: drafted levels, i.e. draft forwards per step
 *   topk      k in [1, 16]: children per expanded node and frontier width
 *   num_keep  m in [0, k + (d-1)k^2]: drafted nodes kept by the rerank; at most 4096 candidates
 *   dtype     of the weights, the embedding and the features; logits are always fp32.  bf16
 *             runs the FC and LM head on the tensor cores with fp32 accumulation and rounds the
 *             FC output to bf16 once; fp32 runs them as fp32 FMA.
 *   fc_weight [h][2h]: columns 0..h-1 multiply the feature, h..2h-1 the token embedding
 *   fc_bias   [h] or NULL (no bias)
 *   lm_head   [V][h], no bias
 *   embedding [V][h]
 */
typedef struct {
    int32_t batch, hidden, vocab, depth, topk, num_keep;
    eagle_dtype dtype;
    const void *fc_weight;
    const void *fc_bias;
    const void *lm_head;
    const void *embedding;
} eagle_tree_config;

typedef struct eagle_tree eagle_tree;

/* Bytes of device workspace a handle for `cfg` needs (0 if cfg is invalid).  Depends on the
 * device current at the call (its SM count sizes the GEMM's split-K scratch). */
EAGLE_API size_t eagle_tree_workspace_bytes(const eagle_tree_config *cfg);

/* Validates cfg, lays the workspace out, builds the TMA descriptors of the weights, clears the
 * workspace's status word and counters (synchronous cudaMemset) and returns a host handle in
 * *out.  The workspace must stay allocated and unused by anything else until destroy.
 * Errors: INVALID_ARG (bad cfg, null/misaligned pointer, workspace too small), UNSUPPORTED,
 * CUDA. */
EAGLE_API eagle_status eagle_tree_init(const eagle_tree_config *cfg, void *d_workspace,
                                       size_t workspace_bytes, eagle_tree **out);

/*
 * EAGLE-1 static tree ("EAGLE notes ch. 04" §10.1 and §12 item 7: EAGLE-1 drafts a tree whose shape
 * is fixed and set by position only; zdszero "EAGLE": one static draft tree, verified with the
 * ancestor-only mask).  The shape is h_spec [num_nodes][2] (host memory): drafted node j (1..N)
 * is (parent, rank), the rank-th most probable draft token (0-based, ties to the lower id) at its
 * parent; parents come first, depth never decreases, ranks are in [0, 16) and distinct among
 * siblings.  cfg->depth must be the shape's depth and cfg->num_keep must be N; cfg->topk is not
 * used.  The handle then works as the dynamic one: eagle_draft_level runs, per level, only the
 * rows of nodes that have children (row top-k of the largest rank + 1, children take their
 * ranked tokens, scores add up as in the dynamic tree); eagle_rerank_build_tree outputs the
 * fixed shape (tokens drafted, parents, depth positions, ancestor mask, scores); verify, node
 * logits, draft extend and the host step are unchanged.  Init copies the shape's constants into
 * the workspace (synchronously).  Errors: INVALID_ARG for a malformed shape or mismatching cfg.
 */
EAGLE_API size_t eagle_tree_workspace_bytes_static(const eagle_tree_config *cfg, int32_t num_nodes,
                                                   const int32_t *h_spec);
EAGLE_API eagle_status eagle_tree_init_static(const eagle_tree_config *cfg, int32_t num_nodes,
                                              const int32_t *h_spec, void *d_ws, size_t ws_bytes,
                                              eagle_tree **out);

/*
 * One draft level ("EAGLE notes ch. 04" §6.1 and §10.3; zdszero "EAGLE-2").
 * level 0 starts a new step: its rows are the B roots, row b = [d_root_feature[b] ||
 *   E[d_root_token[b]]] (d_root_feature [B][h] of cfg.dtype, d_root_token [B]); the root's k
 *   children become candidates 0..k-1 and all k form the first frontier.
 * level l >= 1 must follow level l-1: its B*k rows are the frontier nodes, row b*k+s =
 *   [f^ of the row that produced slot s's node || E[its token]]; child j of slot s becomes
 *   candidate k + (l-1)k^2 + s*k + j with score S = S(slot) + logp_j; the next frontier is
 *   the top-k of the k^2 children by (S descending, candidate ascending).
 * Per row: f^ = FC(row) (rounded to bf16 for bf16), z = LM_head(f^), lse = logsumexp(z),
 *   children = top-k of z by (z descending, token id ascending), logp = z - lse.
 * d_logits_out: optional fp32 [R][V] receiving z of every row (R = B at level 0, else B*k;
 *   4-byte alignment suffices); NULL keeps the logits in the workspace.  The root arguments
 *   are ignored for l >= 1.
 * Errors: INVALID_ARG, STATE (level out of order), CUDA.
 */
EAGLE_API eagle_status eagle_draft_level(eagle_tree *t, int32_t level, const void *d_root_feature,
                                         const int32_t *d_root_token, float *d_logits_out,
                                         eagle_stream_t stream);

/*
 * Draft extend and the next round's root (zdszero "在 SGLang 里": after the verify, the draft runs
 * again over the verified positions with the target's true hidden states and the accepted tokens;
 * the last verified position starts the next round and its top-k is the next round's first
 * level.  "EAGLE notes ch. 04" §6.2 and §12 item 3: the accepted path's true features start the
 * next draft).  Inputs are the verify's outputs and the target's features of every tree node:
 *   d_node_features [B][m+1][h] (cfg.dtype, 16-byte aligned), d_accept_len [B],
 *   d_accept_nodes / d_accept_tokens [B][d+1] (as eagle_verify_greedy / eagle_verify_sample).
 * Row i of request b (i = 0..d) is [F[b][a_j] || E[t_j]], j = min(i, accept_len[b]), a_j the j-th
 * node of the accepted path and t_j the token after it (the bonus for j = accept_len); every row
 * goes through the FC.  The last verified row is also the next round's level-0 row: its f^, LM
 * head, log-softmax + top-k and expand are done here, exactly as eagle_draft_level(t, 0, ...)
 * would with root feature F[b][a_L] and root token t_L, so the next round continues with
 * eagle_draft_level(t, 1, ...).
 *   d_next_root_feature [B][h] (cfg.dtype, 16-byte aligned), d_next_root_token [B]: that root
 *   d_path_fhat  [B][d+1][h] or NULL: the FC output of every row (the draft features along the
 *                accepted path; rows past accept_len repeat its row)
 *   d_logits_out [B][V] fp32 or NULL: the level-0 logits
 * Errors: INVALID_ARG, CUDA; a path entry outside the tree or the vocabulary latches
 * EAGLE_ERR_DEVICE_BOUNDS.
 */
EAGLE_API eagle_status eagle_draft_extend(eagle_tree *t, const void *d_node_features,
                                          const int32_t *d_accept_len, const int32_t *d_accept_nodes,
                                          const int32_t *d_accept_tokens, void *d_next_root_feature,
                                          int32_t *d_next_root_token, void *d_path_fhat,
                                          float *d_logits_out, eagle_stream_t stream);

/*
 * Rerank + tree build, after level d-1 ("EAGLE notes ch. 04" §10.3; zdszero "在 SGLang 里";
 * jsqmd "二、EAGLE-2" steps ① ②).  Per request keeps the top-m candidates by (S descending,
 * candidate ascending) and flattens root + kept nodes, in ascending candidate order, to
 * n = m+1 nodes:
 *   d_tokens    [B][n]  node 0 = the root token, then the kept tokens
 *   d_parents   [B][n]  tree index of the parent, -1 for the root
 *   d_positions [B][n]  depth + d_pos_base[b] (d_pos_base [B] or NULL for 0)
 *   d_mask      [B][n][W] uint32, W = ceil(n/32): bit j (LSB-first, word j/32) of row i is set
 *                       iff j is i or an ancestor of i
 *   d_logscore  [B][n]  S of each node (0 for the root), optional (NULL)
 * Errors: INVALID_ARG, STATE (not after level d-1), CUDA.  A kept node whose parent was not
 * kept (impossible for finite scores) latches EAGLE_ERR_DEVICE_BOUNDS.
 */
EAGLE_API eagle_status eagle_rerank_build_tree(eagle_tree *t, const int32_t *d_pos_base,
                                               int32_t *d_tokens, int32_t *d_parents,
                                               int32_t *d_positions, uint32_t *d_mask,
                                               float *d_logscore, eagle_stream_t stream);

/*
 * Greedy tree verification ("EAGLE notes ch. 04" §6.2; zdszero "Medusa": temperature 0 reduces
 * acceptance to greedy; jsqmd "二、EAGLE-2": accept the longest consistent root path).
 * Works on any tree given as arrays (it does not need the handle's own tree):
 *   d_tokens, d_parents   [B][n], n = m+1, parents before children
 *   d_target_logits       [B][n][V] of target_dtype (EAGLE_F32 or EAGLE_BF16), or NULL
 *   d_target_ids          [B][n] target argmax per node, used when d_target_logits is NULL
 * g_i = argmax_v target[i][v] (ties to the lowest v); from the root, repeatedly accept the child
 * of the current node whose token equals g(current).  Outputs:
 *   d_accept_len    [B]      accepted drafted nodes, 0..d
 *   d_accept_nodes  [B][d+1] tree indices of the accepted path, root first, -1 padded
 *   d_accept_tokens [B][d+1] accepted tokens then the bonus token g(last), -1 padded
 * Errors: INVALID_ARG, CUDA.
 */
EAGLE_API eagle_status eagle_verify_greedy(eagle_tree *t, const int32_t *d_tokens,
                                           const int32_t *d_parents, const void *d_target_logits,
                                           eagle_dtype target_dtype, const int32_t *d_target_ids,
                                           int32_t *d_accept_len, int32_t *d_accept_nodes,
                                           int32_t *d_accept_tokens, eagle_stream_t stream);

/*
 * Draft logits of every node of the tree last built by eagle_rerank_build_tree: node i's own
 * row, [feature that entered i || E[token i]] -> FC -> LM head, i.e. the draft's distribution
 * of i's children.  The root's feature is d_root_feature [B][h] (the same as level 0's).
 * Output d_node_logits [B][n][V] fp32.  Used to synthesise target logits (draft logits plus
 * noise) on the GPU.  Errors: INVALID_ARG, STATE (no tree built yet), CUDA.
 */
EAGLE_API eagle_status eagle_tree_node_logits(eagle_tree *t, const void *d_root_feature,
                                              float *d_node_logits, eagle_stream_t stream);

/*
 * One whole step from host memory: copies the roots (and optional positions) and the target
 * logits to the device, runs levels 0..d-1, the rerank/build and the verify, copies the tree and
 * the verify results back, and returns when they are on the host.  The work runs on a stream of
 * the handle, ordered after everything already queued on `stream`.  The roots go in one copy through a pinned
 * staging image held by the handle; the target logits go on a side stream of the handle while
 * the draft runs (h_target_logits should be pinned for that copy to be asynchronous); the
 * outputs come back in one copy together with the device status word, which the step clears at
 * its start and returns (like eagle_tree_status).  The first call allocates the pinned staging
 * (cudaMallocHost), two streams and three events; eagle_tree_destroy frees them.  The whole
 * sequence is captured once into a CUDA graph (again whenever
 * d_target_staging, target_dtype or the presence of h_pos_base changes) and replayed, with only
 * the target copy's host source updated per call; where capture is not possible the same work
 * is launched directly.
 * d_target_staging is caller-owned device memory of [B][m+1][V] elements of target_dtype that
 * receives h_target_logits.
 *   h_root_feature [B][h] (cfg.dtype), h_root_token [B], h_pos_base [B] or NULL,
 *   h_target_logits [B][m+1][V]; outputs h_tokens/h_parents/h_positions [B][m+1],
 *   h_mask [B][m+1][W] (or NULL), h_accept_len [B], h_accept_tokens [B][d+1].
 * Errors: as the calls it makes.
 */
EAGLE_API eagle_status eagle_tree_step_host(eagle_tree *t, const void *h_root_feature,
                                            const int32_t *h_root_token,
                                            const int32_t *h_pos_base,
                                            const void *h_target_logits, eagle_dtype target_dtype,
                                            void *d_target_staging, int32_t *h_tokens,
                                            int32_t *h_parents, int32_t *h_positions,
                                            uint32_t *h_mask, int32_t *h_accept_len,
                                            int32_t *h_accept_tokens, eagle_stream_t stream);

/* Synchronises `stream`, returns the first error latched by a kernel since the last call
 * (EAGLE_OK if none) and clears the status word. */
EAGLE_API eagle_status eagle_tree_status(eagle_tree *t, eagle_stream_t stream);

/* Frees the host handle (the workspace and the weights stay the caller's). NULL is a no-op. */
EAGLE_API void eagle_tree_destroy(eagle_tree *t);

/* Static, human-readable name of a status code. */
EAGLE_API const char *eagle_status_str(eagle_status s);

/*
 * Where the handle keeps its intermediate state inside the workspace: byte offsets from the
 * workspace base, for tests and debugging.  Rows are padded to r_pad (a multiple of 16).
 *   x            [r_pad][2h] (dtype)      the next level's concatenated rows
 *   fhat         [d][r_pad][h] (dtype)    f^ of every row of every level
 *   logits       [r_pad][V] fp32          z of the last level (when no d_logits_out)
 *   row_ids      [r_pad][k] int32, row_logp [r_pad][k] fp32, row_lse [r_pad] fp32
 *   pool_*       [B][n_cand]  tok int32, S fp32, parent int32 (-1: the root), row int32 (row of
 *                             the producing level whose f^ is the candidate's input feature)
 *   front_cand/front_S [2][B][k]  the frontier, double-buffered by level parity: level l reads
 *                             buffer (l+1)%2... see front_current
 *   node_tok, node_src [B][n] the last tree's tokens and feature rows (fhat row index
 *                             level*r_pad+row, or -1-b for request b's root feature)
 *   target_ids   [B][n] int32 the last verify's target argmax
 */
typedef struct {
    int64_t x, fhat, logits, row_ids, row_logp, row_lse;
    int64_t pool_tok, pool_S, pool_parent, pool_row;
    int64_t front_cand, front_S, node_tok, node_src, target_ids, status;
    int32_t r_pad, n_cand, num_nodes, mask_words;
    int32_t front_current; /* index (0/1) of the buffer holding the frontier for the next level */
    int32_t num_sms;
} eagle_tree_layout;

EAGLE_API eagle_status eagle_tree_get_layout(const eagle_tree *t, eagle_tree_layout *out);

/*
 * Launch accounting and optional timing of the streamed-weight GEMM (the FC and LM-head launches,
 * the path's dominant kernel).  eagle_tree_profile(t, n) creates n pairs of CUDA events (host-side
 * objects, no device memory) and from then on brackets each of the next n GEMM launches of this
 * handle with two events recorded on the launch's stream (not inside a stream capture); n = 0
 * stops and frees them.  eagle_tree_profile_read synchronises on the last event, returns the
 * number of timed launches, their summed duration in ms and their summed algorithmic bytes (the
 * weight matrix, the input rows and the FC's output rows; the LM head's logits are not counted,
 * as the tree only needs each row's top-k and logsumexp), then restarts the count.
 * eagle_tree_launch_count returns how many kernels this handle has launched since init.
 */
EAGLE_API eagle_status eagle_tree_profile(eagle_tree *t, int32_t max_launches);
/* Pauses (enable = 0) or resumes the timing of GEMM launches without freeing the events.  Each
 * timed launch is bracketed by events on its stream, which keeps it from overlapping the
 * previous kernel, so a caller that wants the overlapped throughput times only some steps. */
EAGLE_API eagle_status eagle_tree_profile_enable(eagle_tree *t, int32_t enable);
EAGLE_API eagle_status eagle_tree_profile_read(eagle_tree *t, int32_t *launches, double *total_ms,
                                               double *total_bytes);
/* The same timed launches one by one (at most cap of them, in launch order): duration ms[i],
 * algorithmic bytes[i] (as above), flops[i] = 2 * out_features * in_features * rows, and
 * tag[i] = 2 * level + 0 for the FC or + 1 for the LM head (-1: eagle_tree_node_logits).  *n is
 * the number written; like eagle_tree_profile_read it restarts the count.  All arrays are host
 * memory owned by the caller. */
EAGLE_API eagle_status eagle_tree_profile_list(eagle_tree *t, int32_t cap, int32_t *n, float *ms,
                                               double *bytes, double *flops, int32_t *tag);
EAGLE_API int64_t eagle_tree_launch_count(const eagle_tree *t);
/*
 * Test hook (no counterpart on the pages): shows that a device wait gives up instead of hanging.
 * One thread waits, through the bounded wait that every waiting kernel of this library uses, on
 * an mbarrier nothing arrives on; after limit_ns (1 .. 10^10 ns) it sets the timeout bit in
 * *d_status (a caller-owned int32 in device memory) and returns.  The call synchronises `stream`,
 * reads and clears the word, and returns EAGLE_ERR_DEVICE_TIMEOUT when the bit was set (else
 * EAGLE_OK).  INVALID_ARG for a limit out of range or a null pointer, CUDA on a launch error.
 */
EAGLE_API eagle_status eagle_test_bounded_wait(int64_t limit_ns, int32_t *d_status,
                                               eagle_stream_t stream);
/* 1 when eagle_tree_step_host replays a captured graph, 0 before its first call, -1 when
 * capture failed and the host step launches directly. */
EAGLE_API int32_t eagle_tree_step_graphed(const eagle_tree *t);

/* ------------------------------------------------------------------------------------------ */
/* Stateless kernels of the path, for callers that keep their own state (and for tests).      */
/* ------------------------------------------------------------------------------------------ */

/*
 * Per-row log-softmax and top-k ("EAGLE notes ch. 04" §10.2-§10.3): for each of `rows` rows of
 * d_logits (row r starts at r*ld elements, of dtype EAGLE_F32 or EAGLE_BF16):
 *   d_ids [rows][k]   the k best columns by (value descending, column ascending)
 *   d_vals [rows][k]  value - lse when d_lse is given (log-probabilities), else the raw values
 *   d_lse [rows]      logsumexp of the row (fp32), or NULL
 * k in [1, 16], k <= vocab.  With k = 1 and no d_lse this is the target argmax of verify.
 */
EAGLE_API eagle_status eagle_row_topk(const void *d_logits, eagle_dtype dtype, int32_t rows,
                                      int32_t vocab, int64_t ld, int32_t k, int32_t *d_ids,
                                      float *d_vals, float *d_lse, eagle_stream_t stream);

/*
 * Expand one level for B requests, without features (zdszero "在 SGLang 里": select the top-k of
 * the k^2 children by cumulative score).  Inputs for level 0: d_row_ids / d_row_logp [B][k]
 * (row b = the root of request b).  For level l >= 1: [B*k][k] (row b*k+s = frontier slot s)
 * and the frontier d_front_cand_in / d_front_S_in [B][k].  Writes the level's candidates into
 * the pool d_pool_* [B][n_cand] (n_cand = k + (depth-1)k^2; the candidate numbering of
 * eagle_draft_level) and, when d_front_cand_out is not NULL, the next frontier [B][k].
 * Scores add in fp32; ranks break ties by the lower candidate id.
 */
EAGLE_API eagle_status eagle_expand(int32_t level, int32_t batch, int32_t topk, int32_t depth,
                                    const int32_t *d_row_ids, const float *d_row_logp,
                                    const int32_t *d_front_cand_in, const float *d_front_S_in,
                                    int32_t *d_front_cand_out, float *d_front_S_out,
                                    int32_t *d_pool_tok, float *d_pool_S, int32_t *d_pool_parent,
                                    int32_t *d_pool_row, eagle_stream_t stream);

/*
 * Rerank + tree build from an explicit pool (the arrays eagle_expand writes).  d_root_token [B];
 * outputs as eagle_rerank_build_tree.  d_status: optional int32 word that latches a broken
 * tree (bit 2).
 */
EAGLE_API eagle_status eagle_build_tree(int32_t batch, int32_t topk, int32_t depth,
                                        int32_t num_keep, const int32_t *d_pool_tok,
                                        const float *d_pool_S, const int32_t *d_pool_parent,
                                        const int32_t *d_root_token, const int32_t *d_pos_base,
                                        int32_t *d_tokens, int32_t *d_parents,
                                        int32_t *d_positions, uint32_t *d_mask,
                                        float *d_logscore, int32_t *d_status,
                                        eagle_stream_t stream);

/*
 * The verify walk alone, given the target argmax per node d_target_ids [B][n]: outputs as
 * eagle_verify_greedy.  depth bounds the walk (the accept arrays are [B][depth+1]).
 */
EAGLE_API eagle_status eagle_verify_walk(int32_t batch, int32_t num_nodes, int32_t depth,
                                         const int32_t *d_tokens, const int32_t *d_parents,
                                         const int32_t *d_target_ids, int32_t *d_accept_len,
                                         int32_t *d_accept_nodes, int32_t *d_accept_tokens,
                                         eagle_stream_t stream);

/*
 * Sampling tree verification ("EAGLE notes ch. 04" §6.2 and §7.1; the SGLang note in the summary
 * of tom-jerr's "(EAGLE 1) EAGLE" reading for mode 1).  Stateless; works on any tree given as
 * arrays.  For request b, p_i = softmax(T[b][i] / temperature) and q_i = softmax(Z[b][i] /
 * temperature), where T and Z are the target's and the draft's logits at node i (the
 * distribution of the token after node i; q_i is what node i's children were drafted from).
 * From the root, the children of the current node are tested in ascending tree index:
 *   mode 0 (recursive rejection sampling): child c with token t is accepted iff P(t) > 0 and
 *          u_acc[b][c] * q(t) <= P(t), P being the current distribution (p of the node, then
 *          norm(max(0, P - q)) after each rejected child; an empty residual leaves P as is);
 *   mode 1 (threshold): the first child with p(t) >= threshold is accepted; if none is, P is p
 *          after one rejection step per child.
 * An accepted child becomes the current node (P = its p); the walk stops at depth `depth`, at a
 * leaf, or when no child is accepted, and the bonus token is drawn from P by inverse CDF: the
 * smallest token whose running sum (ascending ids) exceeds u_bonus[b] * sum(P) (else the largest
 * token with P > 0).  All arithmetic is fp32 (the decisions of a double-precision evaluation can
 * differ when a uniform falls within rounding of its threshold).
 *   d_tokens, d_parents [B][n], parents before children, n <= 4097
 *   d_target_logits, d_draft_logits  [B][n][V] fp32 (finite)
 *   d_u_accept [B][n], d_u_bonus [B]  uniforms in [0, 1) drawn by the caller
 *   d_scratch  [B][V] fp32, caller-owned, overwritten
 * Outputs as eagle_verify_greedy.  temperature > 0 (use eagle_verify_greedy for 0).  Errors:
 * INVALID_ARG (sizes, null pointers, temperature, mode), CUDA.  Token ids outside [0, V) are
 * never accepted.
 */
EAGLE_API eagle_status eagle_verify_sample(int32_t batch, int32_t num_nodes, int32_t vocab,
                                           int32_t depth, const int32_t *d_tokens,
                                           const int32_t *d_parents, const float *d_target_logits,
                                           const float *d_draft_logits, float temperature,
                                           int32_t mode, float threshold, const float *d_u_accept,
                                           const float *d_u_bonus, float *d_scratch,
                                           int32_t *d_accept_len, int32_t *d_accept_nodes,
                                           int32_t *d_accept_tokens, eagle_stream_t stream);

/*
 * Streamed-weight GEMM used by the FC and the LM head: Y[r][o] = sum_i W[o][i] X[r][i]
 * (+ bias[o]) for r < rows, o < out_features, with W [out][in] and X [rows][in] bf16 (row
 * strides in elements ldw, ldx; multiples of 8), fp32 accumulation on the tensor cores.  Output
 * Y [rows][ldy]: fp32 when out_bf16 == 0, else bf16 rounded to nearest even.  Needs
 * eagle_linear_workspace_bytes(...) bytes of zero-initialised scratch (d_ws, 256-byte aligned),
 * which it leaves zeroed.  rows in [1, 32768] per call: above 256 the rows are taken in chunks of
 * 256, each a unit of the same launch with every weight tile, so the weights are streamed from
 * memory once for all chunks.
 */
EAGLE_API size_t eagle_linear_workspace_bytes(int32_t out_features, int32_t rows);
EAGLE_API eagle_status eagle_linear_bf16(const void *d_w, int64_t ldw, const void *d_x,
                                         int64_t ldx, const void *d_bias, int32_t out_features,
                                         int32_t in_features, int32_t rows, void *d_y,
                                         int64_t ldy, int32_t out_bf16, void *d_ws,
                                         size_t ws_bytes, eagle_stream_t stream);

/*
 * The draft decoder layer.  zdszero, "在 SGLang 里": after the FC, the draft model runs one Llama
 * decoder layer (its first input_layernorm is the identity; no final norm) and hands its output
 * to the target's LM head.  EAGLE notes ch. 04 §4.1 (the light decoder layer predicts the next
 * feature) and §12.5 (tree attention: each node sees the cached context and its own ancestors).
 * One call runs the layer over the `nodes` tree nodes of each of `batch` requests:
 *   qkv_i = Wqkv x_i (q: heads*head_dim rows, k and v: kv_heads*head_dim rows each);
 *   q_i, k_i rotated by Llama rotate-half RoPE at positions[b][i] (pair (j, j + D/2) turned by
 *   positions * rope_theta^(-2j/D));
 *   o_i = softmax_j(q_i . k_j / sqrt(D)) v_j over the `prefix` cached keys of request b and the
 *   tree nodes that mask row i marks (query head hq reads kv head hq / (heads / kv_heads));
 *   h1 = x_i + Wo o_i;  r = RMSNorm(h1; rms_eps) * w_norm;  [g; u] = Wgu r;
 *   out_i = h1 + Wd (silu(g) * u).
 * Each projection output, the attention output, both residual sums, r and silu(g) * u are bf16
 * (round to nearest even); dot products, the softmax and the norm accumulate in fp32.
 * Weights (bf16, row-major, device, 16-byte aligned): w_qkv [(heads + 2 kv_heads) head_dim]
 * [hidden] (q rows, then k rows, then v rows); w_o [hidden][heads head_dim]; w_norm [hidden];
 * w_gu [2 inter][hidden] (gate rows, then up rows); w_d [hidden][inter].
 * Limits: hidden and inter multiples of 8; head_dim a multiple of 32 and at most 128; heads a
 * multiple of kv_heads; nodes in [1, 4097]; rope_theta > 0; rms_eps >= 0.
 */
typedef struct {
    int32_t hidden, heads, kv_heads, head_dim, inter;
    float rope_theta, rms_eps;
    const void *w_qkv, *w_o, *w_norm, *w_gu, *w_d;
} eagle_decoder_layer_weights;

/*
 * Device scratch bytes for eagle_decoder_layer at these sizes on the current device (0 on
 * unusable sizes or without a device).
 */
EAGLE_API size_t eagle_decoder_layer_workspace_bytes(const eagle_decoder_layer_weights *w,
                                                     int32_t batch, int32_t nodes);
/*
 * Every device array is 16-byte aligned.
 * Inputs (device): d_x [batch][nodes][hidden] bf16; d_k_cache / d_v_cache
 * [batch][prefix][kv_heads][head_dim] bf16, keys already rotated (may be null when prefix == 0);
 * d_positions [batch][nodes] int32; d_mask [batch][nodes][W] uint32 with W = ceil(nodes / 32),
 * bit t of row i set when node t is visible to node i (the tree's ancestor mask).
 * Outputs (device): d_out [batch][nodes][hidden] bf16; d_k_new / d_v_new [batch][nodes][kv_heads]
 * [head_dim] bf16, the tree's rotated keys and values for the caller's cache (both null to skip).
 * d_ws: eagle_decoder_layer_workspace_bytes bytes, 256-byte aligned, zero-filled once before the
 * first call (the GEMM's tile tickets; every call leaves them zero).  A query row with nothing
 * visible gives o = 0.  Calls on one workspace must not overlap.  batch == 0 does nothing.
 * Kernels: the four projections on the streamed-weight tcgen05 GEMM; RoPE (angles reduced in
 * double, one cos/sin per row and pair); tree attention on mma.sync bf16 tensor-core tiles of 64
 * keys with an online softmax (key splits merged by a second kernel when few CTAs); fused
 * residual + RMSNorm; SwiGLU; residual.
 * Returns EAGLE_ERR_INVALID_ARG on bad sizes, null or misaligned pointers or a short workspace,
 * EAGLE_ERR_CUDA when a launch fails.  Asynchronous on `stream`.
 */
EAGLE_API eagle_status eagle_decoder_layer(const eagle_decoder_layer_weights *w, int32_t batch,
                                           int32_t nodes, int32_t prefix, const void *d_x,
                                           const void *d_k_cache, const void *d_v_cache,
                                           const int32_t *d_positions, const uint32_t *d_mask,
                                           void *d_out, void *d_k_new, void *d_v_new, void *d_ws,
                                           size_t ws_bytes, eagle_stream_t stream);

/*
 * The streamed-weight GEMM of eagle_linear_bf16 without caller-provided scratch.  The pages have
 * no counterpart: this is an engineering variant for callers that cannot allocate device memory
 * (code where cudaMalloc is not allowed or not wanted because it synchronises the device and can
 * fail under memory pressure, plug-ins whose host framework owns all device memory, loops that
 * must not allocate per call).  The caller passes only inputs and outputs, with the meaning and
 * layout of eagle_linear_bf16.
 *   - Scratch: a fixed array of eagle_linear_noalloc_scratch_bytes() bytes (about 5 MiB) in this
 *     library's own device memory, held by every GPU that loads the library until exit.  The
 *     first call on a device looks its address up (cudaGetSymbolAddress, with that device
 *     current) and sets the kernel's attributes; make that first call before any stream capture.
 *   - Limits: rows <= 32 and out_features <= 131072; larger sizes return EAGLE_ERR_INVALID_ARG.
 *     The split runs on at most 160 CTAs, which bounds the partial sums the array holds.
 *   - Results: on a GPU with at most 160 SMs the split is the one eagle_linear_bf16 uses, so
 *     the two entry points agree bit for bit; with more SMs the split differs and they agree
 *     within the GEMM's fp32 rounding bound.
 *   - Every call shares the one array: each call clears the tile tickets it needs on its stream
 *     before launching, but calls that overlap on the GPU (other streams, other threads) race.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 */
EAGLE_API size_t eagle_linear_noalloc_scratch_bytes(void);
EAGLE_API eagle_status eagle_linear_bf16_noalloc(const void *d_w, int64_t ldw, const void *d_x,
                                                 int64_t ldx, const void *d_bias,
                                                 int32_t out_features, int32_t in_features,
                                                 int32_t rows, void *d_y, int64_t ldy,
                                                 int32_t out_bf16, eagle_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE_TREE_H */
