// kernels.cuh - host-side interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

namespace eagle {

// Names the calls of one entry point for profilers (NVTX push/pop around the enqueue).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// Launches `kernel` allowing programmatic dependent launch: it may start while the previous
// kernel in the stream is still running.  Every kernel of this library calls griddepcontrol.wait
// before it touches memory a previous kernel may write or read, and launch_dependents early.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same with thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, unsigned cluster, size_t smem,
                               cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------------------------
// Streamed-weight GEMM (FC and LM head), bf16 on the tensor cores:
//   Y[r][o] = sum_i W[o][i] * X[r][i] (+ bias[o]),  r < rows, o < M
// The weight matrix is cut into 128-row tiles and 64-wide k-blocks; the k-blocks of all tiles
// form one stream that is split evenly over a persistent grid (one CTA per SM).  A tile whose
// k-blocks land in more than one CTA is summed in ascending CTA order (deterministic) by the last
// CTA to arrive, by the CTA that finds its partner done, or by a second launch.  Above 16 rows,
// when the tiles pair up, the CTAs run as pairs sharing one M = 256 MMA (.cta_group::2) and the
// stream runs over pairs of tiles.  A row's result is bit-identical among launches of 1-16 rows
// and among launches of 17-256.
// ---------------------------------------------------------------------------------------------
constexpr int kLinearTileM = 128;
constexpr int kLinearTileK = 64;
constexpr int kLinearMaxRows = 256;  // MMA N limit: rows of one row chunk
constexpr int kLinearMaxLaunchRows = 32768;  // rows of one launch (row chunks of kLinearMaxRows)
constexpr int kLinearMaxFixupRows = 16;  // above this, split tiles are summed by their owner or a second launch

struct LinearPlan {
    CUtensorMap tmap_w;  // W [M][K] bf16, box {64, 128}, 128-byte swizzle
    CUtensorMap tmap_x;  // X [rows][K] bf16, box {64, n_tile}, 128-byte swizzle
    CUtensorMap tmap_y;  // Y [rows][ldo], box {128, 32}, no swizzle (valid when y_tma)
    int32_t M, K, rows, n_tile, num_kb, num_tiles, stages, tmem_cols, grid;
    size_t smem_bytes;
    const void *bias;  // [M] bf16 or null
    void *out;         // [rows][ldo]
    int64_t ldo;
    int32_t out_bf16;
    int32_t defer;     // rows > kLinearMaxFixupRows: a second launch sums the split tiles
    int32_t owner_fix; // > 16 rows, at most two CTAs per tile: summed in the launch by its owner
    int32_t pair;      // CTA pairs on .cta_group::2 (clusters of 2; grid = 2 x pairs)
    int32_t num_wtiles;  // weight units of the stream-K split: tiles, or pairs of tiles
    int32_t num_chunks;  // row chunks of n_tile (at most kLinearMaxRows) rows
    int32_t y_tma;     // outputs and partials leave by bulk stores (16-row groups)
    int32_t out_stage_bytes;  // their shared-memory staging
    float *partials;   // [grid][2][n_tile][128]
    int32_t *counters; // [num_tiles][num_chunks], zero before and after
    int32_t *status;
};

// Bytes of split-K scratch (partials) and tile counters a launch with these sizes needs.
size_t linear_partials_bytes(int32_t grid, int32_t n_tile);
size_t linear_counters_bytes(int32_t M, int32_t rows = 1);
int32_t linear_n_tile(int32_t rows);
// Tensor map of a bf16 KV cache [B][P][Hk][D] (D 64 or 128) read in boxes of 64 keys x 64 head
// dims of one kv head, 128-byte swizzled (the tree attention's key and value tiles).
bool encode_kv_cache_map(CUtensorMap *map, const void *cache, int32_t B, int32_t P, int32_t Hk, int32_t D);
// Tensor map of a bf16 matrix [rows][ld] (cols used) in boxes of box_cols x box_rows, 128-byte
// swizzled.
bool encode_bf16_rows_map(CUtensorMap *map, const void *ptr, uint64_t cols, uint64_t rows, uint64_t ld,
                          uint32_t box_cols, uint32_t box_rows);
// CTA pairs of the .cta_group::2 mode that fit on the device at once (0: the mode is off).
int32_t linear_pair_workers(int32_t num_sms);

// Fills `plan` (tensor maps included).  Returns false on an unusable argument (alignment,
// strides, sizes) or when the driver's tensor-map encoder is unavailable.
bool plan_linear_bf16(LinearPlan *plan, const void *w, int64_t ldw, int32_t M, int32_t K,
                      const void *x, int64_t ldx, int32_t rows, const void *bias, void *out,
                      int64_t ldo, int32_t out_bf16, float *partials, int32_t *counters,
                      int32_t *status, int32_t num_sms);
cudaError_t launch_linear_bf16(const LinearPlan &plan, cudaStream_t st);
// Points a plan's output at another buffer of the same layout (re-encodes the output tensor map
// of the TMA stores, or falls back to plain stores when the new buffer does not suit it).
void linear_retarget_out(LinearPlan *plan, void *out);
// One-time per-device kernel attributes (large dynamic shared memory).
cudaError_t prepare_kernels();

// fp32 path (FMA on the CUDA cores), same contract, no scratch.
cudaError_t launch_linear_f32(const float *w, int64_t ldw, const float *x, int64_t ldx,
                              const float *bias, float *y, int64_t ldy, int32_t M, int32_t K,
                              int32_t rows, cudaStream_t st);

// ---------------------------------------------------------------------------------------------
// Per-row log-softmax + top-k (k <= 16), or argmax (k = 1, lse == null): a thread-block cluster
// per row holding the row in registers, or, for at least as many rows as SMs with rows of at
// least 32 KB, one CTA per row streaming it once through shared memory.  `status` (may be null)
// receives kDevTimeout if a streamed copy does not land in time.
// ---------------------------------------------------------------------------------------------
struct ExpandArgs;
// The expand of a draft level run inside the top-k launch: the last row of each request to finish
// (a ticket per request, zero before and after) runs that request's expand.  Only for an expand
// without row copies (x_next null).
struct FusedExpand {
    const ExpandArgs *args;  // null: no fused expand
    int32_t rows_per_req;
    int32_t *tickets;        // [B]
};
cudaError_t launch_row_topk(const void *logits, int32_t is_bf16, int32_t rows, int32_t V,
                            int64_t ld, int32_t k, int32_t *ids, float *vals, float *lse,
                            cudaStream_t st, int32_t *status = nullptr, const FusedExpand *fx = nullptr,
                            bool *fused = nullptr);

// ---------------------------------------------------------------------------------------------
// Tree kernels
// ---------------------------------------------------------------------------------------------
struct ExpandArgs {
    int32_t level, B, k, n_cand, h, V, elem_bytes;
    const int32_t *row_ids;
    const float *row_logp;
    const int32_t *front_cand_in;
    const float *front_S_in;
    int32_t *front_cand_out;  // null on the last level
    float *front_S_out;
    int32_t *pool_tok;
    float *pool_S;
    int32_t *pool_parent;
    int32_t *pool_row;
    const void *fhat;  // this level's f^ rows [.][h], or null (no feature copy)
    const void *emb;   // [V][h]
    void *x_next;      // [B*k][2h], or null
    int32_t *status;
};
cudaError_t launch_expand(const ExpandArgs &a, cudaStream_t st);

struct BuildArgs {
    int32_t B, k, d, m, n_cand, r_pad;
    const int32_t *pool_tok;
    const float *pool_S;
    const int32_t *pool_parent;
    const int32_t *pool_row;  // may be null (node_src then not written)
    const int32_t *root_tok;
    const int32_t *pos_base;  // may be null
    int32_t *tokens, *parents, *positions;
    uint32_t *mask;
    float *logscore;          // may be null
    int32_t *node_tok, *node_src;  // may be null
    int32_t *status;
};
constexpr int32_t kMaxCandidates = 4096;  // rerank pool per request
cudaError_t launch_build_tree(const BuildArgs &a, cudaStream_t st);
cudaError_t prepare_tree_kernels();

// Sampling verification (recursive rejection sampling, mode 0; threshold variant, mode 1); one
// CTA per request; scratch is [B][V] fp32.
cudaError_t launch_verify_sample(int32_t B, int32_t n, int32_t V, int32_t depth, const int32_t *tok,
                                 const int32_t *par, const float *T, const float *Z, float temperature,
                                 int32_t mode, float threshold, const float *u_acc, const float *u_bonus,
                                 float *scratch, int32_t *accept_len, int32_t *accept_nodes,
                                 int32_t *accept_tok, cudaStream_t st);
cudaError_t launch_verify_walk(int32_t B, int32_t n, int32_t d, const int32_t *tok,
                               const int32_t *par, const int32_t *g, int32_t *accept_len,
                               int32_t *accept_nodes, int32_t *accept_tok, cudaStream_t st);
// X[r] = [feature(src[r]) || E[tok[r]]]: src[r] >= 0 is a row of fhat_all, -1-b is row b of
// root_feat; src == null means src[r] = -1-r.
struct GatherArgs {
    int32_t n_rows, h, V, elem_bytes;
    const int32_t *src;
    const int32_t *tok;
    const void *root_feat;
    const void *fhat_all;
    const void *emb;
    void *x;
    int32_t *status;
    int32_t *tok_copy;  // [n_rows] receives tok as given, or null
    int32_t src_rows = 0;   // rows of fhat_all and of root_feat (checking builds), 0: not checked
    int32_t root_rows = 0;
};
cudaError_t launch_gather(const GatherArgs &a, cudaStream_t st);

// Draft extend: path rows [F[b][a_j] || E[t_j]] (j = min(i, accept_len[b])) for i <= d, the next
// round's root (feature, token) and root-token copy; then level 0's f^ rows from the last rows.
struct ExtendArgs {
    int32_t B, d, n, h, V, elem_bytes;
    const void *node_feat;   // [B][n][h]
    const int32_t *accept_len, *accept_nodes, *accept_tok;  // [B], [B][d+1], [B][d+1]
    const void *emb;         // [V][h]
    void *x;                 // [B*(d+1)][2h]
    void *next_feat;         // [B][h]
    int32_t *next_tok;       // [B]
    int32_t *root_tok;       // [B]
    const void *ext_fhat;    // [B*(d+1)][h]
    void *fhat0;             // [B][h] level 0's f^
    void *path_fhat;         // [B][d+1][h] or null
    int32_t *status;
};
cudaError_t launch_extend_gather(const ExtendArgs &a, cudaStream_t st);
cudaError_t launch_extend_select(const ExtendArgs &a, cudaStream_t st);

// EAGLE-1 static tree.  sp points at the per-node constants, field f of node j at sp[f * n + j]:
// 0 parent, 1 rank, 2 depth, 3 index among the nodes of its depth with children (-1: none),
// 4 that index of its parent, 5 level offset of its parent's row ((depth - 1) * r_pad), 6 rows
// per request at its parent's level.
constexpr int kSpPar = 0, kSpRank = 1, kSpDep = 2, kSpEidx = 3, kSpPeidx = 4, kSpSrcOff = 5, kSpEStride = 6;
constexpr int kSpFields = 7;

// Nodes of depth level+1 (first lo, cnt of them): token = the parent row's top-k id at the node's
// rank, score = parent's + that logp; a node with children also gets its row of the next level.
struct StaticExpandArgs {
    int32_t level, B, n, K, E, E_next, h, elem_bytes, lo, cnt, V;
    const int32_t *row_ids;  // [B*E][K]
    const float *row_logp;
    const int32_t *sp;
    int32_t *node_tok;       // [B][n]
    float *node_S;           // [B][n]
    const void *fhat;        // this level's f^ rows [B*E][h]
    const void *emb;
    void *x_next;            // [B*E_next][2h] or null
    int32_t *status;
};
cudaError_t launch_static_expand(const StaticExpandArgs &a, cudaStream_t st);

// The static tree's outputs from the constants and the drafted tokens and scores.
struct StaticBuildArgs {
    int32_t B, n, W;
    const int32_t *sp;
    const uint32_t *sp_mask;   // [n][W]
    const int32_t *root_tok;   // [B]
    const int32_t *pos_base;   // [B] or null
    int32_t *node_tok;         // [B][n]: drafted tokens in, the root written at 0
    const float *node_S;       // [B][n]
    int32_t *node_src;         // [B][n] f^ row feeding each node (node logits)
    int32_t *tokens, *parents, *positions;
    uint32_t *mask;
    float *logscore;           // or null
};
cudaError_t launch_static_build(const StaticBuildArgs &a, cudaStream_t st);

// Test hook: a wait on an mbarrier nothing arrives on, bounded by limit_ns; latches the timeout
// bit in *status.
cudaError_t launch_bounded_wait(uint64_t limit_ns, int32_t *status, cudaStream_t st);

}  // namespace eagle
