// api.cu - the C ABI declared in include/eagle_tree.h: argument checks, workspace layout,
// tensor-map planning and the launch sequence of one draft-tree step.
#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>


#include "../../include/eagle_tree.h"
#include "common.cuh"
#include "kernels.cuh"

using namespace eagle;

namespace {

constexpr int32_t kMaxTopk = 16;
constexpr int32_t kMaxDepth = 32;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// NVTX range over one C-ABI call (host side only; free when no tool is attached).
int32_t round16(int32_t x) { return (x + 15) / 16 * 16; }

struct Layout {
    size_t status, counters, partials, x, fhat, logits, row_ids, row_logp, row_lse;
    size_t pool_tok, pool_S, pool_par, pool_row, front_cand, front_S;
    size_t root_tok, node_tok, node_src, g, node_x, node_fhat, ext_x, ext_fhat;
    size_t xtickets;      // per request: rows of the level whose top-k is done (fused expand)
    // static tree (EAGLE-1) constants per node, and the drafted nodes' scores
    size_t sp_node, sp_mask, node_S;
    size_t st_feat, st_tok, st_pos, st_tokens, st_parents, st_positions, st_mask, st_acc_len,
        st_acc_nodes, st_acc_tok, st_out_end, st_in_end;
    size_t total;
    size_t partials_bytes, counters_bytes;
    int32_t r_pad, n_cand, n_nodes, mask_words, node_chunk, eb;
    int32_t kk;  // entries of each row's top-k (topk; for a static tree, its largest rank + 1)
};

// The shape of an EAGLE-1 static tree ("EAGLE notes ch. 04" §10.1 and §12 item 7: the shape is
// fixed, set by position only): drafted node j (1..N) is (parent, rank), the rank-th most
// probable draft token at its parent.  Everything below is derived on the host once.
struct StaticShape {
    int32_t N = 0, D = 0, K = 0;  // drafted nodes, depth, top-k entries a row needs
    // per node (n = N + 1; the root is node 0): parent, rank, depth, index among the nodes of
    // its depth that have children (-1 if none), and that index of its parent
    std::vector<int32_t> par, rank, dep, eidx, peidx;
    std::vector<int32_t> lo, cnt;  // per depth 0..D: first node and node count
    std::vector<int32_t> E;        // per level 0..D-1: nodes of that depth with children
    std::vector<uint32_t> mask;    // [n][W] ancestor-only, LSB first
};

// Validates a (parent, rank) list: parents first, depth non-decreasing, ranks in [0, 16) and
// below V, distinct ranks among siblings.
bool make_static_shape(int32_t N, const int32_t *spec, int32_t V, StaticShape *s) {
    if (N < 1 || N > kMaxCandidates || !spec) return false;
    const int32_t n = N + 1;
    s->N = N;
    s->par.assign(n, -1);
    s->rank.assign(n, 0);
    s->dep.assign(n, 0);
    s->eidx.assign(n, -1);
    s->peidx.assign(n, -1);
    std::vector<uint32_t> used(n, 0u);  // ranks taken among each node's children
    int32_t K = 1;
    for (int32_t j = 1; j < n; ++j) {
        const int32_t p = spec[2 * (j - 1)], r = spec[2 * (j - 1) + 1];
        if (p < 0 || p >= j || r < 0 || r >= kMaxTopk || r >= V) return false;
        if (used[p] & (1u << r)) return false;
        used[p] |= 1u << r;
        s->par[j] = p;
        s->rank[j] = r;
        s->dep[j] = s->dep[p] + 1;
        if (s->dep[j] < s->dep[j - 1]) return false;
        K = std::max(K, r + 1);
    }
    s->K = K;
    s->D = s->dep[n - 1];
    if (s->D < 1 || s->D > kMaxDepth) return false;
    s->lo.assign(s->D + 1, 0);
    s->cnt.assign(s->D + 1, 0);
    for (int32_t j = n - 1; j >= 0; --j) s->lo[s->dep[j]] = j;
    for (int32_t j = 0; j < n; ++j) ++s->cnt[s->dep[j]];
    s->E.assign(s->D, 0);
    for (int32_t j = 0; j < n; ++j)
        if (used[j] != 0u) s->eidx[j] = s->E[s->dep[j]]++;
    for (int32_t j = 1; j < n; ++j) s->peidx[j] = s->eidx[s->par[j]];
    const int32_t W = (n + 31) / 32;
    s->mask.assign(static_cast<size_t>(n) * W, 0u);
    for (int32_t j = 0; j < n; ++j)
        for (int32_t x = j; x >= 0; x = s->par[x]) s->mask[static_cast<size_t>(j) * W + x / 32] |= 1u << (x % 32);
    return true;
}

bool config_ok(const eagle_tree_config *c) {
    if (!c) return false;
    if (c->batch < 0 || c->hidden < 1 || c->vocab < 1) return false;
    if (c->depth < 1 || c->depth > kMaxDepth) return false;
    if (c->topk < 1 || c->topk > kMaxTopk || c->topk > c->vocab) return false;
    if (c->dtype != EAGLE_F32 && c->dtype != EAGLE_BF16) return false;
    if (c->dtype == EAGLE_BF16 && c->hidden % 8 != 0) return false;
    if (c->dtype == EAGLE_F32 && c->hidden % 4 != 0) return false;
    const int64_t nc = c->topk + static_cast<int64_t>(c->depth - 1) * c->topk * c->topk;
    if (nc > kMaxCandidates) return false;
    if (c->num_keep < 0 || c->num_keep > nc) return false;
    return true;
}

// A static tree's configuration: the shape fixes depth and m (cfg.topk is not used).
bool static_config_ok(const eagle_tree_config *c, const StaticShape &s) {
    if (!c) return false;
    if (c->batch < 0 || c->hidden < 1 || c->vocab < 1) return false;
    if (c->depth != s.D || c->num_keep != s.N) return false;
    if (c->dtype != EAGLE_F32 && c->dtype != EAGLE_BF16) return false;
    if (c->dtype == EAGLE_BF16 && c->hidden % 8 != 0) return false;
    if (c->dtype == EAGLE_F32 && c->hidden % 4 != 0) return false;
    return s.K <= c->vocab;
}

Layout make_layout(const eagle_tree_config *c, int32_t num_sms, const StaticShape *ss = nullptr) {
    Layout L{};
    const int64_t B = c->batch, h = c->hidden, V = c->vocab, d = c->depth;
    const int64_t k = ss ? ss->K : c->topk;
    L.kk = static_cast<int32_t>(k);
    L.eb = (c->dtype == EAGLE_BF16) ? 2 : 4;
    L.n_cand = ss ? 0 : static_cast<int32_t>(k + (d - 1) * k * k);
    L.n_nodes = c->num_keep + 1;
    L.mask_words = (L.n_nodes + 31) / 32;
    int64_t R1 = B * k;
    if (ss) {
        R1 = 0;
        for (int32_t e : ss->E) R1 = std::max<int64_t>(R1, B * e);
    }
    L.r_pad = round16(static_cast<int32_t>(std::max<int64_t>(1, std::max(R1, B))));
    const int64_t node_rows = B * L.n_nodes;
    L.node_chunk = static_cast<int32_t>(node_rows < kLinearMaxRows ? (node_rows > 0 ? node_rows : 1)
                                                                   : kLinearMaxRows);
    const int64_t ext_rows = B * (d + 1);  // draft extend: every verified position of every request
    const int32_t max_rows = static_cast<int32_t>(std::min<int64_t>(
        kLinearMaxRows, std::max<int64_t>(std::max<int64_t>(L.r_pad, L.node_chunk), ext_rows)));
    if (c->dtype == EAGLE_BF16) {
        L.partials_bytes = linear_partials_bytes(num_sms, linear_n_tile(max_rows));
        L.counters_bytes = std::max(linear_counters_bytes(c->hidden), linear_counters_bytes(c->vocab));
    }
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + (bytes ? bytes : 1));
        return at;
    };
    L.status = take(sizeof(int32_t));
    // host-step staging right after the status word: [status | outputs | inputs] is one range, so
    // the host step moves its inputs (and a cleared status word) in one copy and its outputs (with
    // the status word) in another
    L.st_tokens = take(static_cast<size_t>(node_rows) * 4);
    L.st_parents = take(static_cast<size_t>(node_rows) * 4);
    L.st_positions = take(static_cast<size_t>(node_rows) * 4);
    L.st_mask = take(static_cast<size_t>(node_rows) * L.mask_words * 4);
    L.st_acc_len = take(static_cast<size_t>(B) * 4);
    L.st_acc_nodes = take(static_cast<size_t>(B) * (d + 1) * 4);
    L.st_acc_tok = take(static_cast<size_t>(B) * (d + 1) * 4);
    L.st_out_end = o;
    L.st_feat = take(static_cast<size_t>(B) * h * L.eb);
    L.st_tok = take(static_cast<size_t>(B) * 4);
    L.st_pos = take(static_cast<size_t>(B) * 4);
    L.st_in_end = o;
    L.counters = take(L.counters_bytes);
    L.xtickets = take(static_cast<size_t>(B) * 4);  // zero at init, like the tile tickets
    L.partials = take(L.partials_bytes);
    L.x = take(static_cast<size_t>(L.r_pad) * 2 * h * L.eb);
    L.fhat = take(static_cast<size_t>(d) * L.r_pad * h * L.eb);
    L.logits = take(static_cast<size_t>(L.r_pad) * V * 4);
    L.row_ids = take(static_cast<size_t>(L.r_pad) * k * 4);
    L.row_logp = take(static_cast<size_t>(L.r_pad) * k * 4);
    L.row_lse = take(static_cast<size_t>(L.r_pad) * 4);
    L.pool_tok = take(static_cast<size_t>(B) * L.n_cand * 4);
    L.pool_S = take(static_cast<size_t>(B) * L.n_cand * 4);
    L.pool_par = take(static_cast<size_t>(B) * L.n_cand * 4);
    L.pool_row = take(static_cast<size_t>(B) * L.n_cand * 4);
    L.front_cand = take(2 * static_cast<size_t>(B) * k * 4);
    L.front_S = take(2 * static_cast<size_t>(B) * k * 4);
    L.root_tok = take(static_cast<size_t>(B) * 4);
    L.node_tok = take(static_cast<size_t>(node_rows) * 4);
    L.node_src = take(static_cast<size_t>(node_rows) * 4);
    L.g = take(static_cast<size_t>(node_rows) * 4);
    L.node_x = take(static_cast<size_t>(L.node_chunk) * 2 * h * L.eb);
    L.node_fhat = take(static_cast<size_t>(L.node_chunk) * h * L.eb);
    L.ext_x = take(static_cast<size_t>(ext_rows) * 2 * h * L.eb);
    L.ext_fhat = take(static_cast<size_t>(ext_rows) * h * L.eb);
    L.sp_node = take(ss ? static_cast<size_t>(L.n_nodes) * 7 * 4 : 0);
    L.sp_mask = take(ss ? static_cast<size_t>(L.n_nodes) * L.mask_words * 4 : 0);
    L.node_S = take(ss ? static_cast<size_t>(node_rows) * 4 : 0);
    L.total = o;
    return L;
}

int32_t current_num_sms(int32_t *device_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (device_out) *device_out = dev;
    return sms;
}

cudaError_t prepare_device() {
    static std::mutex mu;
    static std::vector<int> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int d : done)
        if (d == dev) return cudaSuccess;
    e = prepare_kernels();
    if (e == cudaSuccess) e = prepare_tree_kernels();
    if (e == cudaSuccess) done.push_back(dev);
    return e;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A GEMM over `rows` rows, split into launches of at most kLinearMaxRows rows.
struct LinearSeq {
    std::vector<LinearPlan> plans;
    std::vector<int32_t> row0;
};

bool plan_seq(LinearSeq *s, const void *w, int64_t ldw, int32_t M, int32_t K, const void *x, int64_t ldx,
              int32_t rows, const void *bias, void *out, int64_t ldo, int32_t out_bf16, int32_t ob,
              float *partials, int32_t *counters, int32_t *status, int32_t num_sms) {
    s->plans.clear();
    s->row0.clear();
    for (int32_t r0 = 0; r0 < rows; r0 += kLinearMaxRows) {
        const int32_t n = std::min(kLinearMaxRows, rows - r0);
        LinearPlan p;
        const uint8_t *xb = reinterpret_cast<const uint8_t *>(x) + static_cast<int64_t>(r0) * ldx * 2;
        uint8_t *yb = reinterpret_cast<uint8_t *>(out) + static_cast<int64_t>(r0) * ldo * ob;
        if (!plan_linear_bf16(&p, w, ldw, M, K, xb, ldx, n, bias, yb, ldo, out_bf16, partials, counters,
                              status, num_sms))
            return false;
        s->plans.push_back(p);
        s->row0.push_back(r0);
    }
    return true;
}

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

struct eagle_tree {
    eagle_tree_config cfg;
    int device = 0;
    int32_t num_sms = 0;
    Layout L;
    uint8_t *ws = nullptr;
    int32_t *status = nullptr, *counters = nullptr;
    float *partials = nullptr;
    int32_t next_level = 0;  // the level eagle_draft_level accepts next (0 is always accepted)
    bool tree_built = false;
    int32_t front_current = 0;
    bool is_static = false;         // EAGLE-1 static tree (shape below) instead of the dynamic one
    StaticShape shape;
    std::vector<LinearSeq> fc, lm;  // per level (bf16 only)
    LinearSeq fc_ext;               // the draft extend's FC over B*(d+1) rows (bf16 only)
    int64_t launches = 0;           // kernels launched by this handle
    std::vector<cudaEvent_t> prof_start, prof_stop;
    std::vector<double> prof_bytes, prof_flops;
    std::vector<int32_t> prof_tag;
    int32_t prof_n = 0;
    bool prof_on = true;
    // host step: pinned image of the workspace range [status, inputs end), a side stream for the
    // target logits and two events (created by the first eagle_tree_step_host)
    uint8_t *h_stage = nullptr;
    cudaStream_t own = nullptr, side = nullptr;  // the step's stream and the target-copy stream
    cudaEvent_t ev_call = nullptr, ev_in = nullptr, ev_t = nullptr;
    // the host step captured as a CUDA graph: replayed while (staging, dtype, positions given)
    // stay the same; only the target copy's host source is patched per call
    cudaGraphExec_t step_exec = nullptr;
    cudaGraphNode_t step_tcopy = nullptr;
    const void *graph_staging = nullptr;
    int32_t graph_dtype = -1;
    bool graph_pos = false, graph_failed = false;
    int64_t graph_launches = 0;  // kernels one replay launches

    ~eagle_tree() {
        free_profile();
        if (step_exec) cudaGraphExecDestroy(step_exec);
        if (ev_call) cudaEventDestroy(ev_call);
        if (ev_in) cudaEventDestroy(ev_in);
        if (ev_t) cudaEventDestroy(ev_t);
        if (side) cudaStreamDestroy(side);
        if (own) cudaStreamDestroy(own);
        if (h_stage) cudaFreeHost(h_stage);
    }
    void free_profile() {
        for (cudaEvent_t e : prof_start) cudaEventDestroy(e);
        for (cudaEvent_t e : prof_stop) cudaEventDestroy(e);
        prof_start.clear();
        prof_stop.clear();
        prof_bytes.clear();
        prof_flops.clear();
        prof_tag.clear();
        prof_n = 0;
    }
    // Launches one GEMM, bracketed by profiling events when enabled.
    // tag: 2 * level + (0 for the FC, 1 for the LM head); -1 outside the draft levels.
    cudaError_t gemm(const LinearPlan &p, cudaStream_t st, int32_t tag) {
        const bool timed = prof_on && prof_n < static_cast<int32_t>(prof_start.size());
        if (timed && cudaEventRecord(prof_start[prof_n], st) != cudaSuccess) return cudaErrorUnknown;
        cudaError_t e = launch_linear_bf16(p, st);
        launches += p.defer ? 2 : 1;
        if (e != cudaSuccess) return e;
        if (timed) {
            if (cudaEventRecord(prof_stop[prof_n], st) != cudaSuccess) return cudaErrorUnknown;
            const double M = p.M, K = p.K, R = p.rows;
            prof_bytes[prof_n] = 2.0 * M * K + 2.0 * R * K + (p.out_bf16 ? 2.0 * R * M : 0.0);
            prof_flops[prof_n] = 2.0 * M * K * R;
            prof_tag[prof_n] = tag;
            ++prof_n;
        }
        return cudaSuccess;
    }
    cudaError_t run(const LinearSeq &s, cudaStream_t st, void *out_override, int64_t ldo, int32_t ob,
                    int32_t tag) {
        for (size_t i = 0; i < s.plans.size(); ++i) {
            LinearPlan p = s.plans[i];
            if (out_override)
                linear_retarget_out(&p, reinterpret_cast<uint8_t *>(out_override) + static_cast<int64_t>(s.row0[i]) * ldo * ob);
            cudaError_t e = gemm(p, st, tag);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }

    template <typename T>
    T *at(size_t off) const {
        return reinterpret_cast<T *>(ws + off);
    }
    void *fhat_level(int32_t l) const {
        return ws + L.fhat + static_cast<size_t>(l) * L.r_pad * cfg.hidden * L.eb;
    }
    int32_t rows_of(int32_t level) const {
        if (is_static) return cfg.batch * shape.E[level];
        return level == 0 ? cfg.batch : cfg.batch * cfg.topk;
    }
};

#define EAGLE_CUDA(expr)                             \
    do {                                             \
        if ((expr) != cudaSuccess) return EAGLE_ERR_CUDA; \
    } while (0)

extern "C" {

const char *eagle_status_str(eagle_status s) {
    switch (s) {
        case EAGLE_OK: return "EAGLE_OK";
        case EAGLE_ERR_INVALID_ARG: return "EAGLE_ERR_INVALID_ARG";
        case EAGLE_ERR_UNSUPPORTED: return "EAGLE_ERR_UNSUPPORTED";
        case EAGLE_ERR_STATE: return "EAGLE_ERR_STATE";
        case EAGLE_ERR_CUDA: return "EAGLE_ERR_CUDA";
        case EAGLE_ERR_DEVICE_TIMEOUT: return "EAGLE_ERR_DEVICE_TIMEOUT";
        case EAGLE_ERR_DEVICE_BOUNDS: return "EAGLE_ERR_DEVICE_BOUNDS";
    }
    return "EAGLE_ERR_UNKNOWN";
}

size_t eagle_tree_workspace_bytes(const eagle_tree_config *cfg) {
    if (!config_ok(cfg)) return 0;
    const int32_t sms = current_num_sms(nullptr);
    if (sms < 1) return 0;
    return make_layout(cfg, sms).total;
}

// Both kinds of handle; `shape` is null for the dynamic tree.
static eagle_status init_handle(const eagle_tree_config *cfg, const StaticShape *shape, void *d_ws, size_t ws_bytes,
                                eagle_tree **out) {
    if (!out) return EAGLE_ERR_INVALID_ARG;
    *out = nullptr;
    if (shape ? !static_config_ok(cfg, *shape) : !config_ok(cfg)) return EAGLE_ERR_INVALID_ARG;
    if (!d_ws || (reinterpret_cast<uintptr_t>(d_ws) % kAlign) != 0) return EAGLE_ERR_INVALID_ARG;
    if (!cfg->fc_weight || !cfg->lm_head || !cfg->embedding) return EAGLE_ERR_INVALID_ARG;
    if (!aligned16(cfg->fc_weight) || !aligned16(cfg->lm_head) || !aligned16(cfg->embedding) ||
        (cfg->fc_bias && !aligned16(cfg->fc_bias)))
        return EAGLE_ERR_INVALID_ARG;
    int dev = 0;
    const int32_t sms = current_num_sms(&dev);
    if (sms < 1) return EAGLE_ERR_CUDA;
    const Layout L = make_layout(cfg, sms, shape);
    if (ws_bytes < L.total) return EAGLE_ERR_INVALID_ARG;
    if (prepare_device() != cudaSuccess) return EAGLE_ERR_CUDA;

    eagle_tree *t = new (std::nothrow) eagle_tree();
    if (!t) return EAGLE_ERR_INVALID_ARG;
    t->cfg = *cfg;
    if (shape) {
        t->is_static = true;
        t->shape = *shape;
    }
    t->device = dev;
    t->num_sms = sms;
    t->L = L;
    t->ws = reinterpret_cast<uint8_t *>(d_ws);
    t->status = t->at<int32_t>(L.status);
    t->counters = t->at<int32_t>(L.counters);
    t->partials = t->at<float>(L.partials);
    // status word, tile counters, pool and frontier start at zero
    if (cudaMemset(t->ws, 0, L.partials) != cudaSuccess ||
        cudaMemset(t->ws + L.pool_tok, 0, L.root_tok - L.pool_tok) != cudaSuccess) {
        delete t;
        return EAGLE_ERR_CUDA;
    }
    const int32_t B = cfg->batch, h = cfg->hidden, V = cfg->vocab, d = cfg->depth;
    if (shape) {
        // the shape's per-node constants and mask, once
        const int32_t n = L.n_nodes;
        std::vector<int32_t> sp(static_cast<size_t>(kSpFields) * n, 0);
        for (int32_t j = 0; j < n; ++j) {
            sp[kSpPar * n + j] = shape->par[j];
            sp[kSpRank * n + j] = shape->rank[j];
            sp[kSpDep * n + j] = shape->dep[j];
            sp[kSpEidx * n + j] = shape->eidx[j];
            sp[kSpPeidx * n + j] = shape->peidx[j];
            sp[kSpSrcOff * n + j] = j == 0 ? 0 : (shape->dep[j] - 1) * L.r_pad;
            sp[kSpEStride * n + j] = j == 0 ? 0 : shape->E[shape->dep[j] - 1];
        }
        if (cudaMemcpy(t->ws + L.sp_node, sp.data(), sp.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(t->ws + L.sp_mask, shape->mask.data(), shape->mask.size() * 4, cudaMemcpyHostToDevice) !=
                cudaSuccess) {
            delete t;
            return EAGLE_ERR_CUDA;
        }
    }
    if (cfg->dtype == EAGLE_BF16 && B > 0) {
        t->fc.resize(d);
        t->lm.resize(d);
        for (int32_t l = 0; l < d; ++l) {
            const int32_t R = t->rows_of(l);
            if (l == 0 && !plan_seq(&t->fc_ext, cfg->fc_weight, 2 * h, h, 2 * h, t->ws + L.ext_x, 2 * h,
                                    B * (d + 1), cfg->fc_bias, t->ws + L.ext_fhat, h, 1, 2, t->partials,
                                    t->counters, t->status, sms)) {
                delete t;
                return EAGLE_ERR_UNSUPPORTED;
            }
            if (!plan_seq(&t->fc[l], cfg->fc_weight, 2 * h, h, 2 * h, t->ws + L.x, 2 * h, R, cfg->fc_bias,
                          t->fhat_level(l), h, 1, 2, t->partials, t->counters, t->status, sms)) {
                delete t;
                return EAGLE_ERR_UNSUPPORTED;
            }
            if (!plan_seq(&t->lm[l], cfg->lm_head, h, V, h, t->fhat_level(l), h, R, nullptr, t->ws + L.logits, V, 0,
                          4, t->partials, t->counters, t->status, sms)) {
                delete t;
                return EAGLE_ERR_UNSUPPORTED;
            }
        }
    }
    *out = t;
    return EAGLE_OK;
}

eagle_status eagle_tree_init(const eagle_tree_config *cfg, void *d_ws, size_t ws_bytes, eagle_tree **out) {
    NvtxRange nvtx_range("eagle_tree_init");
    return init_handle(cfg, nullptr, d_ws, ws_bytes, out);
}

size_t eagle_tree_workspace_bytes_static(const eagle_tree_config *cfg, int32_t num_nodes, const int32_t *h_spec) {
    StaticShape shape;
    if (!cfg || !make_static_shape(num_nodes, h_spec, cfg->vocab, &shape) || !static_config_ok(cfg, shape)) return 0;
    const int32_t sms = current_num_sms(nullptr);
    if (sms < 1) return 0;
    return make_layout(cfg, sms, &shape).total;
}

eagle_status eagle_tree_init_static(const eagle_tree_config *cfg, int32_t num_nodes, const int32_t *h_spec,
                                    void *d_ws, size_t ws_bytes, eagle_tree **out) {
    NvtxRange nvtx_range("eagle_tree_init_static");
    if (out) *out = nullptr;
    StaticShape shape;
    if (!cfg || !make_static_shape(num_nodes, h_spec, cfg->vocab, &shape)) return EAGLE_ERR_INVALID_ARG;
    return init_handle(cfg, &shape, d_ws, ws_bytes, out);
}

void eagle_tree_destroy(eagle_tree *t) { delete t; }

eagle_status eagle_tree_get_layout(const eagle_tree *t, eagle_tree_layout *o) {
    if (!t || !o) return EAGLE_ERR_INVALID_ARG;
    const Layout &L = t->L;
    o->x = L.x;
    o->fhat = L.fhat;
    o->logits = L.logits;
    o->row_ids = L.row_ids;
    o->row_logp = L.row_logp;
    o->row_lse = L.row_lse;
    o->pool_tok = L.pool_tok;
    o->pool_S = L.pool_S;
    o->pool_parent = L.pool_par;
    o->pool_row = L.pool_row;
    o->front_cand = L.front_cand;
    o->front_S = L.front_S;
    o->node_tok = L.node_tok;
    o->node_src = L.node_src;
    o->target_ids = L.g;
    o->status = L.status;
    o->r_pad = L.r_pad;
    o->n_cand = L.n_cand;
    o->num_nodes = L.n_nodes;
    o->mask_words = L.mask_words;
    o->front_current = t->front_current;
    o->num_sms = t->num_sms;
    return EAGLE_OK;
}

// The part of a draft level after its FC: LM head on the level's f^ rows, log-softmax + top-k of
// every row, expand (pool, next frontier, next level's rows), and the level bookkeeping.
static eagle_status level_tail(eagle_tree *t, int32_t level, float *d_logits_out, cudaStream_t st) {
    const eagle_tree_config &c = t->cfg;
    const Layout &L = t->L;
    const int32_t B = c.batch, h = c.hidden, V = c.vocab, k = c.topk, d = c.depth;
    const int32_t R = t->rows_of(level);
    void *x = t->ws + L.x;
    void *fh = t->fhat_level(level);
    const bool bf16 = c.dtype == EAGLE_BF16;
    // LM head: z = W_lm f^
    float *lg = d_logits_out ? d_logits_out : t->at<float>(L.logits);
    if (bf16) {
        EAGLE_CUDA(t->run(t->lm[level], st, d_logits_out, V, 4, 2 * level + 1));
    } else {
        EAGLE_CUDA(launch_linear_f32(reinterpret_cast<const float *>(c.lm_head), h,
                                     reinterpret_cast<const float *>(fh), h, nullptr, lg, V, V, h, R, st));
        ++t->launches;
    }
    // log-softmax + top-k children of every row
    if (t->is_static) {
        EAGLE_CUDA(launch_row_topk(lg, 0, R, V, V, L.kk, t->at<int32_t>(L.row_ids), t->at<float>(L.row_logp),
                                   t->at<float>(L.row_lse), st, t->status));
        ++t->launches;
        // the nodes of depth level+1 take their ranked tokens; those with children get their rows
        const StaticShape &sh = t->shape;
        const bool more_s = level < d - 1;
        StaticExpandArgs se{};
        se.level = level;
        se.B = B;
        se.n = L.n_nodes;
        se.K = L.kk;
        se.E = sh.E[level];
        se.E_next = more_s ? sh.E[level + 1] : 0;
        se.h = h;
        se.elem_bytes = L.eb;
        se.lo = sh.lo[level + 1];
        se.cnt = sh.cnt[level + 1];
        se.V = V;
        se.row_ids = t->at<int32_t>(L.row_ids);
        se.row_logp = t->at<float>(L.row_logp);
        se.sp = t->at<int32_t>(L.sp_node);
        se.node_tok = t->at<int32_t>(L.node_tok);
        se.node_S = t->at<float>(L.node_S);
        se.fhat = fh;
        se.emb = c.embedding;
        se.x_next = more_s ? x : nullptr;
        se.status = t->status;
        EAGLE_CUDA(launch_static_expand(se, st));
        ++t->launches;
        t->next_level = level + 1;
        return EAGLE_OK;
    }
    // expand: pool, next frontier, next level's rows
    const size_t fstride = static_cast<size_t>(B) * k;
    ExpandArgs e{};
    e.level = level;
    e.B = B;
    e.k = k;
    e.n_cand = L.n_cand;
    e.h = h;
    e.V = V;
    e.elem_bytes = L.eb;
    e.row_ids = t->at<int32_t>(L.row_ids);
    e.row_logp = t->at<float>(L.row_logp);
    const int32_t in_buf = (level + 1) % 2, out_buf = level % 2;
    e.front_cand_in = level == 0 ? nullptr : t->at<int32_t>(L.front_cand) + in_buf * fstride;
    e.front_S_in = level == 0 ? nullptr : t->at<float>(L.front_S) + in_buf * fstride;
    const bool more = level < d - 1;
    e.front_cand_out = more ? t->at<int32_t>(L.front_cand) + out_buf * fstride : nullptr;
    e.front_S_out = more ? t->at<float>(L.front_S) + out_buf * fstride : nullptr;
    e.pool_tok = t->at<int32_t>(L.pool_tok);
    e.pool_S = t->at<float>(L.pool_S);
    e.pool_parent = t->at<int32_t>(L.pool_par);
    e.pool_row = t->at<int32_t>(L.pool_row);
    e.fhat = fh;
    e.emb = c.embedding;
    e.x_next = more ? x : nullptr;
    e.status = t->status;
    // the top-k launch runs the expand too when it copies no rows (its last finishing row of each
    // request does the request's expand)
    FusedExpand fx{nullptr, 0, nullptr};
    if (e.x_next == nullptr) fx = FusedExpand{&e, level == 0 ? 1 : k, t->at<int32_t>(L.xtickets)};
    bool fused = false;
    EAGLE_CUDA(launch_row_topk(lg, 0, R, V, V, L.kk, t->at<int32_t>(L.row_ids), t->at<float>(L.row_logp),
                               t->at<float>(L.row_lse), st, t->status, &fx, &fused));
    ++t->launches;
    if (!fused) {
        EAGLE_CUDA(launch_expand(e, st));
        ++t->launches;
    }
    t->next_level = level + 1;
    if (more) t->front_current = out_buf;
    return EAGLE_OK;
}

eagle_status eagle_draft_level(eagle_tree *t, int32_t level, const void *d_root_feature,
                               const int32_t *d_root_token, float *d_logits_out, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_draft_level");
    if (!t) return EAGLE_ERR_INVALID_ARG;
    const eagle_tree_config &c = t->cfg;
    if (level < 0 || level >= c.depth) return EAGLE_ERR_INVALID_ARG;
    if (level != 0 && level != t->next_level) return EAGLE_ERR_STATE;
    const int32_t B = c.batch, h = c.hidden, V = c.vocab;
    if (B == 0) {
        t->tree_built = false;
        t->next_level = level + 1;
        return EAGLE_OK;
    }
    if (level == 0 && (!d_root_feature || !d_root_token || !aligned16(d_root_feature)))
        return EAGLE_ERR_INVALID_ARG;
    if (d_logits_out && (reinterpret_cast<uintptr_t>(d_logits_out) & 3u) != 0) return EAGLE_ERR_INVALID_ARG;
    t->tree_built = false;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const Layout &L = t->L;
    const int32_t R = t->rows_of(level);
    void *x = t->ws + L.x;
    void *fh = t->fhat_level(level);
    const bool bf16 = c.dtype == EAGLE_BF16;

    if (level == 0) {
        // the gather also keeps a copy of the root tokens for the tree build (a kernel rather than
        // a copy, so that the launch chain stays programmatic)
        GatherArgs g{B, h, V, L.eb, nullptr, d_root_token, d_root_feature, t->ws + L.fhat, c.embedding, x,
                     t->status, t->at<int32_t>(L.root_tok)};
        EAGLE_CUDA(launch_gather(g, st));
        ++t->launches;
    }
    // FC: f^ = W_fc [f || e(t)] + b
    if (bf16) {
        EAGLE_CUDA(t->run(t->fc[level], st, nullptr, h, 2, 2 * level));
    } else {
        EAGLE_CUDA(launch_linear_f32(reinterpret_cast<const float *>(c.fc_weight), 2 * h,
                                     reinterpret_cast<const float *>(x), 2 * h,
                                     reinterpret_cast<const float *>(c.fc_bias), reinterpret_cast<float *>(fh),
                                     h, h, 2 * h, R, st));
        ++t->launches;
    }
    return level_tail(t, level, d_logits_out, st);
}

eagle_status eagle_draft_extend(eagle_tree *t, const void *d_node_features, const int32_t *d_accept_len,
                               const int32_t *d_accept_nodes, const int32_t *d_accept_tokens,
                               void *d_next_root_feature, int32_t *d_next_root_token, void *d_path_fhat,
                               float *d_logits_out, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_draft_extend");
    if (!t) return EAGLE_ERR_INVALID_ARG;
    const eagle_tree_config &c = t->cfg;
    const int32_t B = c.batch, h = c.hidden, d = c.depth;
    if (B == 0) {
        t->tree_built = false;
        t->next_level = 1;
        return EAGLE_OK;
    }
    if (!d_node_features || !d_accept_len || !d_accept_nodes || !d_accept_tokens || !d_next_root_feature ||
        !d_next_root_token)
        return EAGLE_ERR_INVALID_ARG;
    if (!aligned16(d_node_features) || !aligned16(d_next_root_feature) || (d_path_fhat && !aligned16(d_path_fhat)))
        return EAGLE_ERR_INVALID_ARG;
    if (d_logits_out && (reinterpret_cast<uintptr_t>(d_logits_out) & 3u) != 0) return EAGLE_ERR_INVALID_ARG;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const Layout &L = t->L;
    t->tree_built = false;
    ExtendArgs e{};
    e.B = B;
    e.d = d;
    e.n = L.n_nodes;
    e.h = h;
    e.V = c.vocab;
    e.elem_bytes = L.eb;
    e.node_feat = d_node_features;
    e.accept_len = d_accept_len;
    e.accept_nodes = d_accept_nodes;
    e.accept_tok = d_accept_tokens;
    e.emb = c.embedding;
    e.x = t->ws + L.ext_x;
    e.next_feat = d_next_root_feature;
    e.next_tok = d_next_root_token;
    e.root_tok = t->at<int32_t>(L.root_tok);
    e.ext_fhat = t->ws + L.ext_fhat;
    e.fhat0 = t->fhat_level(0);
    e.path_fhat = d_path_fhat;
    e.status = t->status;
    // rows of every verified position, their FC, and level 0's rows out of the last ones
    EAGLE_CUDA(launch_extend_gather(e, st));
    ++t->launches;
    if (c.dtype == EAGLE_BF16) {
        EAGLE_CUDA(t->run(t->fc_ext, st, nullptr, h, 2, -1));
    } else {
        EAGLE_CUDA(launch_linear_f32(reinterpret_cast<const float *>(c.fc_weight), 2 * h,
                                     reinterpret_cast<const float *>(t->ws + L.ext_x), 2 * h,
                                     reinterpret_cast<const float *>(c.fc_bias),
                                     reinterpret_cast<float *>(t->ws + L.ext_fhat), h, h, 2 * h, B * (d + 1), st));
        ++t->launches;
    }
    EAGLE_CUDA(launch_extend_select(e, st));
    ++t->launches;
    // the rest of level 0 (LM head, top-k, expand): the next round continues at level 1
    t->next_level = 0;
    return level_tail(t, 0, d_logits_out, st);
}

eagle_status eagle_rerank_build_tree(eagle_tree *t, const int32_t *d_pos_base, int32_t *d_tokens,
                                     int32_t *d_parents, int32_t *d_positions, uint32_t *d_mask,
                                     float *d_logscore, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_rerank_build_tree");
    if (!t) return EAGLE_ERR_INVALID_ARG;
    if (t->next_level != t->cfg.depth) return EAGLE_ERR_STATE;
    const eagle_tree_config &c = t->cfg;
    if (c.batch == 0) {
        t->tree_built = true;
        return EAGLE_OK;
    }
    if (!d_tokens || !d_parents || !d_positions || !d_mask) return EAGLE_ERR_INVALID_ARG;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    const Layout &L = t->L;
    if (t->is_static) {
        // the shape is fixed: copy it, with the drafted tokens and scores
        StaticBuildArgs sb{};
        sb.B = c.batch;
        sb.n = L.n_nodes;
        sb.W = L.mask_words;
        sb.sp = t->at<int32_t>(L.sp_node);
        sb.sp_mask = t->at<uint32_t>(L.sp_mask);
        sb.root_tok = t->at<int32_t>(L.root_tok);
        sb.pos_base = d_pos_base;
        sb.node_tok = t->at<int32_t>(L.node_tok);
        sb.node_S = t->at<float>(L.node_S);
        sb.node_src = t->at<int32_t>(L.node_src);
        sb.tokens = d_tokens;
        sb.parents = d_parents;
        sb.positions = d_positions;
        sb.mask = d_mask;
        sb.logscore = d_logscore;
        EAGLE_CUDA(launch_static_build(sb, reinterpret_cast<cudaStream_t>(stream)));
        ++t->launches;
        t->tree_built = true;
        return EAGLE_OK;
    }
    BuildArgs a{};
    a.B = c.batch;
    a.k = c.topk;
    a.d = c.depth;
    a.m = c.num_keep;
    a.n_cand = L.n_cand;
    a.r_pad = L.r_pad;
    a.pool_tok = t->at<int32_t>(L.pool_tok);
    a.pool_S = t->at<float>(L.pool_S);
    a.pool_parent = t->at<int32_t>(L.pool_par);
    a.pool_row = t->at<int32_t>(L.pool_row);
    a.root_tok = t->at<int32_t>(L.root_tok);
    a.pos_base = d_pos_base;
    a.tokens = d_tokens;
    a.parents = d_parents;
    a.positions = d_positions;
    a.mask = d_mask;
    a.logscore = d_logscore;
    a.node_tok = t->at<int32_t>(L.node_tok);
    a.node_src = t->at<int32_t>(L.node_src);
    a.status = t->status;
    EAGLE_CUDA(launch_build_tree(a, reinterpret_cast<cudaStream_t>(stream)));
    ++t->launches;
    t->tree_built = true;
    return EAGLE_OK;
}

eagle_status eagle_verify_greedy(eagle_tree *t, const int32_t *d_tokens, const int32_t *d_parents,
                                 const void *d_target_logits, eagle_dtype target_dtype,
                                 const int32_t *d_target_ids, int32_t *d_accept_len, int32_t *d_accept_nodes,
                                 int32_t *d_accept_tokens, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_verify_greedy");
    if (!t) return EAGLE_ERR_INVALID_ARG;
    const eagle_tree_config &c = t->cfg;
    if (c.batch == 0) return EAGLE_OK;
    if (!d_tokens || !d_parents || !d_accept_len || !d_accept_nodes || !d_accept_tokens)
        return EAGLE_ERR_INVALID_ARG;
    if (!d_target_logits && !d_target_ids) return EAGLE_ERR_INVALID_ARG;
    if (d_target_logits && target_dtype != EAGLE_F32 && target_dtype != EAGLE_BF16)
        return EAGLE_ERR_INVALID_ARG;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int32_t n = t->L.n_nodes;
    const int32_t *g = d_target_ids;
    if (d_target_logits) {
        int32_t *gw = t->at<int32_t>(t->L.g);
        EAGLE_CUDA(launch_row_topk(d_target_logits, target_dtype == EAGLE_BF16, c.batch * n, c.vocab, c.vocab, 1,
                                   gw, nullptr, nullptr, st, t->status));
        ++t->launches;
        g = gw;
    }
    EAGLE_CUDA(launch_verify_walk(c.batch, n, c.depth, d_tokens, d_parents, g, d_accept_len, d_accept_nodes,
                                  d_accept_tokens, st));
    ++t->launches;
    return EAGLE_OK;
}

eagle_status eagle_tree_node_logits(eagle_tree *t, const void *d_root_feature, float *d_node_logits,
                                    eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_tree_node_logits");
    if (!t) return EAGLE_ERR_INVALID_ARG;
    if (!t->tree_built) return EAGLE_ERR_STATE;
    const eagle_tree_config &c = t->cfg;
    if (c.batch == 0) return EAGLE_OK;
    if (!d_root_feature || !d_node_logits || !aligned16(d_root_feature)) return EAGLE_ERR_INVALID_ARG;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const Layout &L = t->L;
    const int32_t h = c.hidden, V = c.vocab;
    const int32_t total = c.batch * L.n_nodes;
    const bool bf16 = c.dtype == EAGLE_BF16;
    void *nx = t->ws + L.node_x;
    void *nf = t->ws + L.node_fhat;
    for (int32_t r0 = 0; r0 < total; r0 += L.node_chunk) {
        const int32_t rows = std::min(L.node_chunk, total - r0);
        GatherArgs g{rows, h, V, L.eb, t->at<int32_t>(L.node_src) + r0, t->at<int32_t>(L.node_tok) + r0,
                     d_root_feature, t->ws + L.fhat, c.embedding, nx, t->status, nullptr};
        g.src_rows = c.depth * L.r_pad;  // node sources index every level's f^ rows, or a root
        g.root_rows = c.batch;
        EAGLE_CUDA(launch_gather(g, st));
        ++t->launches;
        float *out = d_node_logits + static_cast<int64_t>(r0) * V;
        if (bf16) {
            LinearSeq fc, lm;
            if (!plan_seq(&fc, c.fc_weight, 2 * h, h, 2 * h, nx, 2 * h, rows, c.fc_bias, nf, h, 1, 2, t->partials,
                          t->counters, t->status, t->num_sms) ||
                !plan_seq(&lm, c.lm_head, h, V, h, nf, h, rows, nullptr, out, V, 0, 4, t->partials, t->counters,
                          t->status, t->num_sms))
                return EAGLE_ERR_UNSUPPORTED;
            EAGLE_CUDA(t->run(fc, st, nullptr, h, 2, -1));
            EAGLE_CUDA(t->run(lm, st, nullptr, V, 4, -1));
        } else {
            EAGLE_CUDA(launch_linear_f32(reinterpret_cast<const float *>(c.fc_weight), 2 * h,
                                         reinterpret_cast<const float *>(nx), 2 * h,
                                         reinterpret_cast<const float *>(c.fc_bias), reinterpret_cast<float *>(nf), h,
                                         h, 2 * h, rows, st));
            EAGLE_CUDA(launch_linear_f32(reinterpret_cast<const float *>(c.lm_head), h,
                                         reinterpret_cast<const float *>(nf), h, nullptr, out, V, V, h, rows, st));
            t->launches += 2;
        }
    }
    return EAGLE_OK;
}

eagle_status eagle_tree_status(eagle_tree *t, eagle_stream_t stream) {
    if (!t) return EAGLE_ERR_INVALID_ARG;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t word = 0;
    EAGLE_CUDA(cudaMemcpyAsync(&word, t->status, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    EAGLE_CUDA(cudaMemsetAsync(t->status, 0, sizeof(int32_t), st));
    EAGLE_CUDA(cudaStreamSynchronize(st));
    if (word & kDevTimeout) return EAGLE_ERR_DEVICE_TIMEOUT;
    if (word & (kDevBounds | kDevTree)) return EAGLE_ERR_DEVICE_BOUNDS;
    return EAGLE_OK;
}

// The device side of one host step, enqueued on `st`: one copy of [status = 0 | outputs | roots]
// from the pinned image, the target logits on the side stream, levels 0..d-1, rerank/build,
// verify (after the target copy), one copy of [status | outputs] back to the image.
static eagle_status enqueue_host_step(eagle_tree *t, const void *h_target_logits, eagle_dtype target_dtype,
                                      void *d_target_staging, bool with_pos, cudaStream_t st) {
    const eagle_tree_config &c = t->cfg;
    const Layout &L = t->L;
    const int32_t B = c.batch, n = L.n_nodes;
    const size_t tbytes = static_cast<size_t>(B) * n * c.vocab * (target_dtype == EAGLE_BF16 ? 2 : 4);
    eagle_stream_t stream = reinterpret_cast<eagle_stream_t>(st);
    EAGLE_CUDA(cudaMemcpyAsync(t->ws + L.status, t->h_stage, L.st_in_end - L.status, cudaMemcpyHostToDevice, st));
    EAGLE_CUDA(cudaEventRecord(t->ev_in, st));
    EAGLE_CUDA(cudaStreamWaitEvent(t->side, t->ev_in, 0));
    EAGLE_CUDA(cudaMemcpyAsync(d_target_staging, h_target_logits, tbytes, cudaMemcpyHostToDevice, t->side));
    EAGLE_CUDA(cudaEventRecord(t->ev_t, t->side));
    eagle_status s;
    for (int32_t l = 0; l < c.depth; ++l) {
        s = eagle_draft_level(t, l, t->ws + L.st_feat, t->at<int32_t>(L.st_tok), nullptr, stream);
        if (s != EAGLE_OK) return s;
    }
    s = eagle_rerank_build_tree(t, with_pos ? t->at<int32_t>(L.st_pos) : nullptr, t->at<int32_t>(L.st_tokens),
                                t->at<int32_t>(L.st_parents), t->at<int32_t>(L.st_positions),
                                t->at<uint32_t>(L.st_mask), nullptr, stream);
    if (s != EAGLE_OK) return s;
    EAGLE_CUDA(cudaStreamWaitEvent(st, t->ev_t, 0));
    s = eagle_verify_greedy(t, t->at<int32_t>(L.st_tokens), t->at<int32_t>(L.st_parents), d_target_staging,
                            target_dtype, nullptr, t->at<int32_t>(L.st_acc_len), t->at<int32_t>(L.st_acc_nodes),
                            t->at<int32_t>(L.st_acc_tok), stream);
    if (s != EAGLE_OK) return s;
    EAGLE_CUDA(cudaMemcpyAsync(t->h_stage, t->ws + L.status, L.st_out_end - L.status, cudaMemcpyDeviceToHost, st));
    return EAGLE_OK;
}

// Captures enqueue_host_step into a graph; on any failure the handle stays on eager launches.
static void capture_host_step(eagle_tree *t, const void *h_target_logits, eagle_dtype target_dtype,
                              void *d_target_staging, bool with_pos, cudaStream_t st) {
    if (t->step_exec) {
        cudaGraphExecDestroy(t->step_exec);
        t->step_exec = nullptr;
    }
    const bool prof = t->prof_on;
    t->prof_on = false;  // no profiling events inside the graph
    const int64_t l0 = t->launches;
    cudaGraph_t g = nullptr;
    bool ok = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
    if (ok) {
        const eagle_status s = enqueue_host_step(t, h_target_logits, target_dtype, d_target_staging, with_pos, st);
        const cudaError_t e = cudaStreamEndCapture(st, &g);
        ok = s == EAGLE_OK && e == cudaSuccess && g != nullptr;
    }
    t->prof_on = prof;
    t->graph_launches = t->launches - l0;
    t->launches = l0;
    cudaGraphNode_t tcopy = nullptr;
    if (ok) {
        size_t nn = 0;
        ok = cudaGraphGetNodes(g, nullptr, &nn) == cudaSuccess && nn > 0;
        std::vector<cudaGraphNode_t> nodes(nn);
        if (ok) ok = cudaGraphGetNodes(g, nodes.data(), &nn) == cudaSuccess;
        for (size_t i = 0; ok && i < nn; ++i) {
            cudaGraphNodeType ty;
            if (cudaGraphNodeGetType(nodes[i], &ty) != cudaSuccess || ty != cudaGraphNodeTypeMemcpy) continue;
            cudaMemcpy3DParms mp = {};
            if (cudaGraphMemcpyNodeGetParams(nodes[i], &mp) == cudaSuccess && mp.dstPtr.ptr == d_target_staging)
                tcopy = nodes[i];
        }
        ok = ok && tcopy != nullptr;
    }
    cudaGraphExec_t ex = nullptr;
    if (ok) ok = cudaGraphInstantiate(&ex, g, 0) == cudaSuccess;
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();  // a failed capture leaves nothing behind
    if (!ok) {
        t->graph_failed = true;
        return;
    }
    t->step_exec = ex;
    t->step_tcopy = tcopy;
    t->graph_staging = d_target_staging;
    t->graph_dtype = target_dtype;
    t->graph_pos = with_pos;
}

eagle_status eagle_tree_step_host(eagle_tree *t, const void *h_root_feature, const int32_t *h_root_token,
                                  const int32_t *h_pos_base, const void *h_target_logits, eagle_dtype target_dtype,
                                  void *d_target_staging, int32_t *h_tokens, int32_t *h_parents,
                                  int32_t *h_positions, uint32_t *h_mask, int32_t *h_accept_len,
                                  int32_t *h_accept_tokens, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_tree_step_host");
    if (!t) return EAGLE_ERR_INVALID_ARG;
    const eagle_tree_config &c = t->cfg;
    if (c.batch == 0) return EAGLE_OK;
    if (!h_root_feature || !h_root_token || !h_target_logits || !d_target_staging || !h_tokens || !h_parents ||
        !h_positions || !h_accept_len || !h_accept_tokens)
        return EAGLE_ERR_INVALID_ARG;
    if (target_dtype != EAGLE_F32 && target_dtype != EAGLE_BF16) return EAGLE_ERR_INVALID_ARG;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const Layout &L = t->L;
    const int32_t B = c.batch, n = L.n_nodes, d = c.depth;
    const size_t tbytes = static_cast<size_t>(B) * n * c.vocab * (target_dtype == EAGLE_BF16 ? 2 : 4);
    if (!t->h_stage) {
        if (cudaMallocHost(&t->h_stage, L.st_in_end - L.status) != cudaSuccess) {
            t->h_stage = nullptr;
            return EAGLE_ERR_CUDA;
        }
        EAGLE_CUDA(cudaStreamCreateWithFlags(&t->own, cudaStreamNonBlocking));
        EAGLE_CUDA(cudaStreamCreateWithFlags(&t->side, cudaStreamNonBlocking));
        EAGLE_CUDA(cudaEventCreateWithFlags(&t->ev_call, cudaEventDisableTiming));
        EAGLE_CUDA(cudaEventCreateWithFlags(&t->ev_in, cudaEventDisableTiming));
        EAGLE_CUDA(cudaEventCreateWithFlags(&t->ev_t, cudaEventDisableTiming));
    }
    uint8_t *hs = t->h_stage;
    const auto at = [&](size_t off) { return hs + (off - L.status); };
    // the roots, and a cleared status word, into the pinned image
    *reinterpret_cast<int32_t *>(hs) = 0;
    std::memcpy(at(L.st_feat), h_root_feature, static_cast<size_t>(B) * c.hidden * L.eb);
    std::memcpy(at(L.st_tok), h_root_token, sizeof(int32_t) * B);
    if (h_pos_base) std::memcpy(at(L.st_pos), h_pos_base, sizeof(int32_t) * B);
    const bool with_pos = h_pos_base != nullptr;
    // The step runs on the handle's own stream, after everything already queued on the caller's
    // (the legacy default stream cannot be captured into a graph; the call synchronises anyway).
    EAGLE_CUDA(cudaEventRecord(t->ev_call, st));
    st = t->own;
    EAGLE_CUDA(cudaStreamWaitEvent(st, t->ev_call, 0));
    if (!t->graph_failed &&
        (!t->step_exec || t->graph_staging != d_target_staging || t->graph_dtype != target_dtype ||
         t->graph_pos != with_pos))
        capture_host_step(t, h_target_logits, target_dtype, d_target_staging, with_pos, st);
    bool replayed = false;
    if (t->step_exec && !t->graph_failed) {
        // a source the graph cannot take (another kind of host memory) runs this call eagerly
        if (cudaGraphExecMemcpyNodeSetParams1D(t->step_exec, t->step_tcopy, d_target_staging, h_target_logits,
                                               tbytes, cudaMemcpyHostToDevice) == cudaSuccess) {
            EAGLE_CUDA(cudaGraphLaunch(t->step_exec, st));
            t->launches += t->graph_launches;
            replayed = true;
        } else {
            cudaGetLastError();
        }
    }
    if (!replayed) {
        const eagle_status s0 = enqueue_host_step(t, h_target_logits, target_dtype, d_target_staging, with_pos, st);
        if (s0 != EAGLE_OK) return s0;
    }
    EAGLE_CUDA(cudaStreamSynchronize(st));
    const size_t nb = sizeof(int32_t) * B * n;
    std::memcpy(h_tokens, at(L.st_tokens), nb);
    std::memcpy(h_parents, at(L.st_parents), nb);
    std::memcpy(h_positions, at(L.st_positions), nb);
    if (h_mask) std::memcpy(h_mask, at(L.st_mask), nb * L.mask_words);
    std::memcpy(h_accept_len, at(L.st_acc_len), sizeof(int32_t) * B);
    std::memcpy(h_accept_tokens, at(L.st_acc_tok), sizeof(int32_t) * B * (d + 1));
    const int32_t word = *reinterpret_cast<const int32_t *>(hs);
    if (word != 0) {
        EAGLE_CUDA(cudaMemset(t->status, 0, sizeof(int32_t)));  // read and cleared, as eagle_tree_status
        if (word & kDevTimeout) return EAGLE_ERR_DEVICE_TIMEOUT;
        return EAGLE_ERR_DEVICE_BOUNDS;
    }
    return EAGLE_OK;
}

eagle_status eagle_tree_profile(eagle_tree *t, int32_t max_launches) {
    if (!t || max_launches < 0) return EAGLE_ERR_INVALID_ARG;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    t->free_profile();
    for (int32_t i = 0; i < max_launches; ++i) {
        cudaEvent_t a, b;
        if (cudaEventCreate(&a) != cudaSuccess) return EAGLE_ERR_CUDA;
        if (cudaEventCreate(&b) != cudaSuccess) {
            cudaEventDestroy(a);
            return EAGLE_ERR_CUDA;
        }
        t->prof_start.push_back(a);
        t->prof_stop.push_back(b);
        t->prof_bytes.push_back(0.0);
        t->prof_flops.push_back(0.0);
        t->prof_tag.push_back(-1);
    }
    return EAGLE_OK;
}

eagle_status eagle_tree_profile_read(eagle_tree *t, int32_t *launches, double *total_ms, double *total_bytes) {
    if (!t || !launches || !total_ms || !total_bytes) return EAGLE_ERR_INVALID_ARG;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    double ms = 0.0, bytes = 0.0;
    if (t->prof_n > 0) EAGLE_CUDA(cudaEventSynchronize(t->prof_stop[t->prof_n - 1]));
    for (int32_t i = 0; i < t->prof_n; ++i) {
        float e = 0.0f;
        EAGLE_CUDA(cudaEventElapsedTime(&e, t->prof_start[i], t->prof_stop[i]));
        ms += e;
        bytes += t->prof_bytes[i];
    }
    *launches = t->prof_n;
    *total_ms = ms;
    *total_bytes = bytes;
    t->prof_n = 0;
    return EAGLE_OK;
}

eagle_status eagle_tree_profile_list(eagle_tree *t, int32_t cap, int32_t *n, float *ms, double *bytes,
                                     double *flops, int32_t *tag) {
    if (!t || !n || cap < 0 || (cap > 0 && (!ms || !bytes || !flops || !tag))) return EAGLE_ERR_INVALID_ARG;
    DeviceGuard guard(t->device);
    if (!guard.ok) return EAGLE_ERR_CUDA;
    if (t->prof_n > 0) EAGLE_CUDA(cudaEventSynchronize(t->prof_stop[t->prof_n - 1]));
    const int32_t m = std::min(cap, t->prof_n);
    for (int32_t i = 0; i < m; ++i) {
        EAGLE_CUDA(cudaEventElapsedTime(&ms[i], t->prof_start[i], t->prof_stop[i]));
        bytes[i] = t->prof_bytes[i];
        flops[i] = t->prof_flops[i];
        tag[i] = t->prof_tag[i];
    }
    *n = m;
    t->prof_n = 0;
    return EAGLE_OK;
}

eagle_status eagle_tree_profile_enable(eagle_tree *t, int32_t enable) {
    if (!t) return EAGLE_ERR_INVALID_ARG;
    t->prof_on = enable != 0;
    return EAGLE_OK;
}

int64_t eagle_tree_launch_count(const eagle_tree *t) { return t ? t->launches : 0; }

eagle_status eagle_test_bounded_wait(int64_t limit_ns, int32_t *d_status, eagle_stream_t stream) {
    if (!d_status || limit_ns < 1 || limit_ns > 10000000000ll) return EAGLE_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    EAGLE_CUDA(launch_bounded_wait(static_cast<uint64_t>(limit_ns), d_status, st));
    int32_t word = 0;
    EAGLE_CUDA(cudaMemcpyAsync(&word, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    EAGLE_CUDA(cudaMemsetAsync(d_status, 0, sizeof(int32_t), st));
    EAGLE_CUDA(cudaStreamSynchronize(st));
    return (word & kDevTimeout) ? EAGLE_ERR_DEVICE_TIMEOUT : EAGLE_OK;
}

int32_t eagle_tree_step_graphed(const eagle_tree *t) {
    if (!t) return 0;
    if (t->graph_failed) return -1;
    return t->step_exec ? 1 : 0;
}

// ------------------------------------------------------------------------------------------------
// Stateless entry points
// ------------------------------------------------------------------------------------------------

eagle_status eagle_row_topk(const void *d_logits, eagle_dtype dtype, int32_t rows, int32_t vocab, int64_t ld,
                            int32_t k, int32_t *d_ids, float *d_vals, float *d_lse, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_row_topk");
    if (rows < 0 || vocab < 1 || ld < vocab || k < 1 || k > kMaxTopk || k > vocab) return EAGLE_ERR_INVALID_ARG;
    if (dtype != EAGLE_F32 && dtype != EAGLE_BF16) return EAGLE_ERR_INVALID_ARG;
    if (rows == 0) return EAGLE_OK;
    if (!d_logits || !d_ids) return EAGLE_ERR_INVALID_ARG;
    EAGLE_CUDA(launch_row_topk(d_logits, dtype == EAGLE_BF16, rows, vocab, ld, k, d_ids, d_vals, d_lse,
                               reinterpret_cast<cudaStream_t>(stream)));
    return EAGLE_OK;
}

eagle_status eagle_expand(int32_t level, int32_t batch, int32_t topk, int32_t depth, const int32_t *d_row_ids,
                          const float *d_row_logp, const int32_t *d_front_cand_in, const float *d_front_S_in,
                          int32_t *d_front_cand_out, float *d_front_S_out, int32_t *d_pool_tok, float *d_pool_S,
                          int32_t *d_pool_parent, int32_t *d_pool_row, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_expand");
    if (batch < 0 || topk < 1 || topk > kMaxTopk || depth < 1 || depth > kMaxDepth || level < 0 || level >= depth)
        return EAGLE_ERR_INVALID_ARG;
    const int64_t nc = topk + static_cast<int64_t>(depth - 1) * topk * topk;
    if (nc > kMaxCandidates) return EAGLE_ERR_INVALID_ARG;
    if (batch == 0) return EAGLE_OK;
    if (!d_row_ids || !d_row_logp || !d_pool_tok || !d_pool_S || !d_pool_parent || !d_pool_row)
        return EAGLE_ERR_INVALID_ARG;
    if (level > 0 && (!d_front_cand_in || !d_front_S_in)) return EAGLE_ERR_INVALID_ARG;
    if ((d_front_cand_out == nullptr) != (d_front_S_out == nullptr)) return EAGLE_ERR_INVALID_ARG;
    ExpandArgs e{};
    e.level = level;
    e.B = batch;
    e.k = topk;
    e.n_cand = static_cast<int32_t>(nc);
    e.h = 0;
    e.V = INT32_MAX;
    e.elem_bytes = 2;
    e.row_ids = d_row_ids;
    e.row_logp = d_row_logp;
    e.front_cand_in = d_front_cand_in;
    e.front_S_in = d_front_S_in;
    e.front_cand_out = d_front_cand_out;
    e.front_S_out = d_front_S_out;
    e.pool_tok = d_pool_tok;
    e.pool_S = d_pool_S;
    e.pool_parent = d_pool_parent;
    e.pool_row = d_pool_row;
    EAGLE_CUDA(launch_expand(e, reinterpret_cast<cudaStream_t>(stream)));
    return EAGLE_OK;
}

eagle_status eagle_build_tree(int32_t batch, int32_t topk, int32_t depth, int32_t num_keep, const int32_t *d_pool_tok,
                              const float *d_pool_S, const int32_t *d_pool_parent, const int32_t *d_root_token,
                              const int32_t *d_pos_base, int32_t *d_tokens, int32_t *d_parents, int32_t *d_positions,
                              uint32_t *d_mask, float *d_logscore, int32_t *d_status, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_build_tree");
    if (batch < 0 || topk < 1 || topk > kMaxTopk || depth < 1 || depth > kMaxDepth) return EAGLE_ERR_INVALID_ARG;
    const int64_t nc = topk + static_cast<int64_t>(depth - 1) * topk * topk;
    if (nc > kMaxCandidates || num_keep < 0 || num_keep > nc) return EAGLE_ERR_INVALID_ARG;
    if (batch == 0) return EAGLE_OK;
    if (!d_pool_tok || !d_pool_S || !d_pool_parent || !d_root_token || !d_tokens || !d_parents || !d_positions ||
        !d_mask)
        return EAGLE_ERR_INVALID_ARG;
    if (prepare_device() != cudaSuccess) return EAGLE_ERR_CUDA;
    BuildArgs a{};
    a.B = batch;
    a.k = topk;
    a.d = depth;
    a.m = num_keep;
    a.n_cand = static_cast<int32_t>(nc);
    a.pool_tok = d_pool_tok;
    a.pool_S = d_pool_S;
    a.pool_parent = d_pool_parent;
    a.root_tok = d_root_token;
    a.pos_base = d_pos_base;
    a.tokens = d_tokens;
    a.parents = d_parents;
    a.positions = d_positions;
    a.mask = d_mask;
    a.logscore = d_logscore;
    a.status = d_status;
    EAGLE_CUDA(launch_build_tree(a, reinterpret_cast<cudaStream_t>(stream)));
    return EAGLE_OK;
}

eagle_status eagle_verify_walk(int32_t batch, int32_t num_nodes, int32_t depth, const int32_t *d_tokens,
                               const int32_t *d_parents, const int32_t *d_target_ids, int32_t *d_accept_len,
                               int32_t *d_accept_nodes, int32_t *d_accept_tokens, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_verify_walk");
    if (batch < 0 || num_nodes < 1 || depth < 0) return EAGLE_ERR_INVALID_ARG;
    if (batch == 0) return EAGLE_OK;
    if (!d_tokens || !d_parents || !d_target_ids || !d_accept_len || !d_accept_nodes || !d_accept_tokens)
        return EAGLE_ERR_INVALID_ARG;
    EAGLE_CUDA(launch_verify_walk(batch, num_nodes, depth, d_tokens, d_parents, d_target_ids, d_accept_len,
                                  d_accept_nodes, d_accept_tokens, reinterpret_cast<cudaStream_t>(stream)));
    return EAGLE_OK;
}

eagle_status eagle_verify_sample(int32_t batch, int32_t num_nodes, int32_t vocab, int32_t depth,
                                 const int32_t *d_tokens, const int32_t *d_parents, const float *d_target_logits,
                                 const float *d_draft_logits, float temperature, int32_t mode, float threshold,
                                 const float *d_u_accept, const float *d_u_bonus, float *d_scratch,
                                 int32_t *d_accept_len, int32_t *d_accept_nodes, int32_t *d_accept_tokens,
                                 eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_verify_sample");
    if (batch < 0 || num_nodes < 1 || num_nodes > kMaxCandidates + 1 || vocab < 1 || depth < 0 || depth > 64)
        return EAGLE_ERR_INVALID_ARG;
    if (!(temperature > 0.0f) || !(temperature < INFINITY) || (mode != 0 && mode != 1)) return EAGLE_ERR_INVALID_ARG;
    if (batch == 0) return EAGLE_OK;
    if (!d_tokens || !d_parents || !d_target_logits || !d_draft_logits || !d_u_accept || !d_u_bonus ||
        !d_scratch || !d_accept_len || !d_accept_nodes || !d_accept_tokens)
        return EAGLE_ERR_INVALID_ARG;
    EAGLE_CUDA(launch_verify_sample(batch, num_nodes, vocab, depth, d_tokens, d_parents, d_target_logits,
                                    d_draft_logits, temperature, mode, threshold, d_u_accept, d_u_bonus, d_scratch,
                                    d_accept_len, d_accept_nodes, d_accept_tokens,
                                    reinterpret_cast<cudaStream_t>(stream)));
    return EAGLE_OK;
}

size_t eagle_linear_workspace_bytes(int32_t out_features, int32_t rows) {
    if (out_features < 1 || rows < 1 || rows > kLinearMaxLaunchRows) return 0;
    const int32_t sms = current_num_sms(nullptr);
    if (sms < 1) return 0;
    return align_up(linear_counters_bytes(out_features, rows)) +
           linear_partials_bytes(sms, linear_n_tile(std::min(rows, kLinearMaxRows)));
}

eagle_status eagle_linear_bf16(const void *d_w, int64_t ldw, const void *d_x, int64_t ldx, const void *d_bias,
                               int32_t out_features, int32_t in_features, int32_t rows, void *d_y, int64_t ldy,
                               int32_t out_bf16, void *d_ws, size_t ws_bytes, eagle_stream_t stream) {
    NvtxRange nvtx_range("eagle_linear_bf16");
    if (out_features < 1 || in_features < 1 || rows < 1 || rows > kLinearMaxLaunchRows) return EAGLE_ERR_INVALID_ARG;
    if (!d_w || !d_x || !d_y || !d_ws) return EAGLE_ERR_INVALID_ARG;
    if (ldw < in_features || ldx < in_features || ldy < out_features) return EAGLE_ERR_INVALID_ARG;
    if (ldw % 8 != 0 || ldx % 8 != 0 || !aligned16(d_w) || !aligned16(d_x)) return EAGLE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_ws) % kAlign) != 0) return EAGLE_ERR_INVALID_ARG;
    if (ws_bytes < eagle_linear_workspace_bytes(out_features, rows)) return EAGLE_ERR_INVALID_ARG;
    const int32_t sms = current_num_sms(nullptr);
    if (sms < 1) return EAGLE_ERR_CUDA;
    if (prepare_device() != cudaSuccess) return EAGLE_ERR_CUDA;
    int32_t *counters = reinterpret_cast<int32_t *>(d_ws);
    float *partials = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(d_ws) +
                                                align_up(linear_counters_bytes(out_features, rows)));
    LinearPlan p;
    if (!plan_linear_bf16(&p, d_w, ldw, out_features, in_features, d_x, ldx, rows, d_bias, d_y, ldy, out_bf16,
                          partials, counters, nullptr, sms))
        return EAGLE_ERR_INVALID_ARG;
    EAGLE_CUDA(launch_linear_bf16(p, reinterpret_cast<cudaStream_t>(stream)));
    return EAGLE_OK;
}

}  // extern "C"
