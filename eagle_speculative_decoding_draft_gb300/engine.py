"""Python face of the draft-tree engine: argument marshalling over the C ABI, nothing else.

Every step of the path runs in the CUDA library (``lib/libeagle_tree.so``); this module only
passes torch tensors' device pointers and the current CUDA stream.  PyTorch provides device
memory and streams.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import EAGLE_BF16, EAGLE_F32, check


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return EAGLE_BF16
    if dt == torch.float32:
        return EAGLE_F32
    raise TypeError(f"unsupported dtype {dt}")


def _need(t, name, dtype=None, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


class EagleTree:
    """One draft-tree engine handle (see include/eagle_tree.h).

    Weights are borrowed: the tensors must stay alive while the handle is used (the handle keeps
    references).  w_fc [h][2h], b_fc [h] or None, w_lm [V][h], emb [V][h], all bf16 or all fp32.
    """

    def __init__(self, w_fc, b_fc, w_lm, emb, batch: int, depth: int, topk: int, num_keep: int,
                 static_spec=None, workspace=None):
        """static_spec: None for the dynamic EAGLE-2 tree, or an EAGLE-1 static shape as
        [(parent, rank), ...] for drafted nodes 1..N (then depth and num_keep must be its depth
        and N; topk is not used).  workspace: a uint8 CUDA tensor of at least the workspace size
        (256-byte aligned) to use instead of a fresh one."""
        self.lib = _lib.load()
        dt = w_fc.dtype
        for name, t in (("w_fc", w_fc), ("w_lm", w_lm), ("emb", emb)):
            _need(t, name, dt)
        if b_fc is not None:
            _need(b_fc, "b_fc", dt)
        self.device = w_fc.device
        self.dtype = dt
        self.hidden = int(w_fc.shape[0])
        self.vocab = int(w_lm.shape[0])
        self.batch, self.depth, self.topk, self.num_keep = batch, depth, topk, num_keep
        self.num_nodes = num_keep + 1
        self.mask_words = (self.num_nodes + 31) // 32
        self._keep = (w_fc, b_fc, w_lm, emb)
        self.cfg = _lib.TreeConfig(batch, self.hidden, self.vocab, depth, topk, num_keep,
                                   _dtype_code(dt), w_fc.data_ptr(),
                                   None if b_fc is None else b_fc.data_ptr(), w_lm.data_ptr(),
                                   emb.data_ptr())
        self.static_spec = None
        if static_spec is not None:
            import numpy as np
            sp = np.ascontiguousarray(np.asarray(static_spec, dtype=np.int32).reshape(-1, 2))
            self.static_spec = sp
            spp = sp.ctypes.data_as(ctypes.c_void_p)
        with torch.cuda.device(self.device):
            if self.static_spec is None:
                nbytes = self.lib.eagle_tree_workspace_bytes(ctypes.byref(self.cfg))
            else:
                nbytes = self.lib.eagle_tree_workspace_bytes_static(ctypes.byref(self.cfg), sp.shape[0], spp)
            if nbytes == 0:
                raise ValueError("invalid draft-tree configuration")
            if workspace is None:
                self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            else:
                if workspace.dtype != torch.uint8 or workspace.numel() < nbytes:
                    raise ValueError(f"workspace must be uint8 with at least {nbytes} bytes")
                self.workspace = _need(workspace, "workspace")
            h = ctypes.c_void_p()
            if self.static_spec is None:
                check(self.lib.eagle_tree_init(ctypes.byref(self.cfg),
                                               ctypes.c_void_p(self.workspace.data_ptr()), nbytes,
                                               ctypes.byref(h)), "eagle_tree_init")
            else:
                check(self.lib.eagle_tree_init_static(ctypes.byref(self.cfg), sp.shape[0], spp,
                                                      ctypes.c_void_p(self.workspace.data_ptr()), nbytes,
                                                      ctypes.byref(h)), "eagle_tree_init_static")
        self._h = h
        self.layout = _lib.TreeLayout()
        check(self.lib.eagle_tree_get_layout(self._h, ctypes.byref(self.layout)),
              "eagle_tree_get_layout")

    # -- lifetime ---------------------------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            self.lib.eagle_tree_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _s(self, stream):
        return _stream(self.device, stream)

    # -- the step ---------------------------------------------------------------------------
    def draft_level(self, level: int, root_feature=None, root_token=None, logits_out=None,
                    stream=None):
        if level == 0:
            _need(root_feature, "root_feature", self.dtype)
            _need(root_token, "root_token", torch.int32)
        if logits_out is not None:
            _need(logits_out, "logits_out", torch.float32)
        check(self.lib.eagle_draft_level(self._h, level, _ptr(root_feature), _ptr(root_token),
                                         _ptr(logits_out), self._s(stream)),
              f"eagle_draft_level({level})")

    def new_tree_outputs(self):
        B, n, W = self.batch, self.num_nodes, self.mask_words
        i32 = dict(dtype=torch.int32, device=self.device)
        return {"tokens": torch.empty(B, n, **i32), "parents": torch.empty(B, n, **i32),
                "positions": torch.empty(B, n, **i32),
                "mask": torch.empty(B, n, W, **i32),
                "logscore": torch.empty(B, n, dtype=torch.float32, device=self.device)}

    def rerank_build_tree(self, pos_base=None, out=None, stream=None):
        out = out or self.new_tree_outputs()
        if pos_base is not None:
            _need(pos_base, "pos_base", torch.int32)
        check(self.lib.eagle_rerank_build_tree(
            self._h, _ptr(pos_base), _ptr(out["tokens"]), _ptr(out["parents"]),
            _ptr(out["positions"]), _ptr(out["mask"]), _ptr(out.get("logscore")),
            self._s(stream)), "eagle_rerank_build_tree")
        return out

    def new_verify_outputs(self):
        i32 = dict(dtype=torch.int32, device=self.device)
        return {"accept_len": torch.empty(self.batch, **i32),
                "accept_nodes": torch.empty(self.batch, self.depth + 1, **i32),
                "accept_tokens": torch.empty(self.batch, self.depth + 1, **i32)}

    def verify_greedy(self, tokens, parents, target_logits=None, target_ids=None, out=None,
                      stream=None):
        out = out or self.new_verify_outputs()
        code = EAGLE_F32
        if target_logits is not None:
            _need(target_logits, "target_logits")
            code = _dtype_code(target_logits.dtype)
        check(self.lib.eagle_verify_greedy(
            self._h, _ptr(_need(tokens, "tokens", torch.int32)),
            _ptr(_need(parents, "parents", torch.int32)), _ptr(target_logits), code,
            _ptr(target_ids), _ptr(out["accept_len"]), _ptr(out["accept_nodes"]),
            _ptr(out["accept_tokens"]), self._s(stream)), "eagle_verify_greedy")
        return out

    def node_logits(self, root_feature, out=None, stream=None):
        if out is None:
            out = torch.empty(self.batch, self.num_nodes, self.vocab, dtype=torch.float32,
                              device=self.device)
        check(self.lib.eagle_tree_node_logits(self._h, _ptr(_need(root_feature, "root_feature",
                                                                  self.dtype)),
                                              _ptr(out), self._s(stream)),
              "eagle_tree_node_logits")
        return out

    def status(self, stream=None):
        check(self.lib.eagle_tree_status(self._h, self._s(stream)), "eagle_tree_status")

    def draft(self, root_feature, root_token, pos_base=None, tree_out=None, logits_out=None,
              stream=None):
        """Levels 0..d-1 then the rerank/build; returns the tree tensors."""
        for level in range(self.depth):
            self.draft_level(level, root_feature, root_token,
                             None if logits_out is None else logits_out[level], stream)
        return self.rerank_build_tree(pos_base, tree_out, stream)

    def extend(self, node_features, accept_len, accept_nodes, accept_tokens, path_fhat=None,
               logits_out=None, stream=None):
        """Draft extend after a verify: the FC over every verified position of the accepted
        paths and the next round's level 0 (continue with draft_level(1, ...)).  Returns the next
        round's root (feature, token)."""
        B, h = self.batch, self.hidden
        feat = torch.empty(B, h, dtype=node_features.dtype, device=self.device)
        tok = torch.empty(B, dtype=torch.int32, device=self.device)
        check(self.lib.eagle_draft_extend(
            self._h, _ptr(_need(node_features, "node_features")), _ptr(accept_len),
            _ptr(accept_nodes), _ptr(accept_tokens), _ptr(feat), _ptr(tok), _ptr(path_fhat),
            _ptr(logits_out), self._s(stream)), "eagle_draft_extend")
        return feat, tok

    def step(self, root_feature, root_token, target_logits, pos_base=None, tree_out=None,
             verify_out=None, stream=None):
        """One whole draft-tree step on device tensors: draft, rerank/build, greedy verify."""
        tree = self.draft(root_feature, root_token, pos_base, tree_out, None, stream)
        ver = self.verify_greedy(tree["tokens"], tree["parents"], target_logits, None,
                                 verify_out, stream)
        return tree, ver

    def step_host(self, root_feature, root_token, target_logits, target_staging, host_out,
                  pos_base=None, stream=None):
        """One whole step from host (pinned) tensors, through eagle_tree_step_host; the results
        land in host_out's tensors ("tokens", "parents", "positions", "mask", "accept_len",
        "accept_tokens").  Synchronises the stream."""
        code = _dtype_code(target_logits.dtype)
        check(self.lib.eagle_tree_step_host(
            self._h, _ptr(root_feature), _ptr(root_token), _ptr(pos_base), _ptr(target_logits),
            code, _ptr(target_staging), _ptr(host_out["tokens"]), _ptr(host_out["parents"]),
            _ptr(host_out["positions"]), _ptr(host_out.get("mask")),
            _ptr(host_out["accept_len"]), _ptr(host_out["accept_tokens"]), self._s(stream)),
            "eagle_tree_step_host")
        return host_out

    # -- accounting ---------------------------------------------------------------------------
    def profile(self, max_launches: int):
        """Time the next max_launches GEMM launches with CUDA events (0 stops)."""
        check(self.lib.eagle_tree_profile(self._h, int(max_launches)), "eagle_tree_profile")

    def profile_enable(self, on: bool):
        """Pause or resume the GEMM launch timing (the events stay allocated)."""
        check(self.lib.eagle_tree_profile_enable(self._h, int(bool(on))), "eagle_tree_profile_enable")

    def profile_read(self):
        """(launches, total_ms, total_algorithmic_bytes) of the GEMM launches timed so far."""
        n = ctypes.c_int32()
        ms = ctypes.c_double()
        by = ctypes.c_double()
        check(self.lib.eagle_tree_profile_read(self._h, ctypes.byref(n), ctypes.byref(ms),
                                               ctypes.byref(by)), "eagle_tree_profile_read")
        return n.value, ms.value, by.value

    def profile_list(self, cap: int):
        """The GEMM launches timed so far, one dict per launch: ms, bytes, flops, level and
        kind ('fc' or 'lm_head'; level -1 for node_logits)."""
        n = ctypes.c_int32()
        ms = (ctypes.c_float * max(cap, 1))()
        by = (ctypes.c_double * max(cap, 1))()
        fl = (ctypes.c_double * max(cap, 1))()
        tg = (ctypes.c_int32 * max(cap, 1))()
        check(self.lib.eagle_tree_profile_list(self._h, int(cap), ctypes.byref(n), ms, by, fl, tg),
              "eagle_tree_profile_list")
        out = []
        for i in range(n.value):
            t = tg[i]
            out.append({"ms": float(ms[i]), "bytes": float(by[i]), "flops": float(fl[i]),
                        "level": t // 2 if t >= 0 else -1,
                        "kind": "lm_head" if (t >= 0 and t % 2) else "fc"})
        return out

    def step_graphed(self) -> int:
        """1: step_host replays a captured graph; 0: not yet; -1: capture failed and step_host
        launches directly."""
        return int(self.lib.eagle_tree_step_graphed(self._h))

    def launch_count(self) -> int:
        return int(self.lib.eagle_tree_launch_count(self._h))

    # -- introspection ----------------------------------------------------------------------
    def views(self):
        """Torch views of the handle's intermediate state inside the workspace."""
        L = self.layout
        ws = self.workspace
        B, k, d, h, V = self.batch, self.topk, self.depth, self.hidden, self.vocab
        eb = 2 if self.dtype == torch.bfloat16 else 4

        def view(off, shape, dtype, esize):
            n = 1
            for s in shape:
                n *= s
            return ws[off:off + n * esize].view(dtype).view(*shape)

        rp = L.r_pad
        nc, n = L.n_cand, L.num_nodes
        return {
            "x": view(L.x, (rp, 2 * h), self.dtype, eb),
            "fhat": view(L.fhat, (d, rp, h), self.dtype, eb),
            "logits": view(L.logits, (rp, V), torch.float32, 4),
            "row_ids": view(L.row_ids, (rp, k), torch.int32, 4),
            "row_logp": view(L.row_logp, (rp, k), torch.float32, 4),
            "row_lse": view(L.row_lse, (rp,), torch.float32, 4),
            "pool_tok": view(L.pool_tok, (B, nc), torch.int32, 4),
            "pool_S": view(L.pool_S, (B, nc), torch.float32, 4),
            "pool_parent": view(L.pool_parent, (B, nc), torch.int32, 4),
            "pool_row": view(L.pool_row, (B, nc), torch.int32, 4),
            "front_cand": view(L.front_cand, (2, B, k), torch.int32, 4),
            "front_S": view(L.front_S, (2, B, k), torch.float32, 4),
            "node_tok": view(L.node_tok, (B, n), torch.int32, 4),
            "node_src": view(L.node_src, (B, n), torch.int32, 4),
            "target_ids": view(L.target_ids, (B, n), torch.int32, 4),
        }


# ----------------------------------------------------------------------------------------------
# Stateless kernels
# ----------------------------------------------------------------------------------------------

def row_topk(logits, k: int, with_lse: bool = True, stream=None):
    """Per-row top-k of a [rows][V] (or [rows][ld] view) fp32/bf16 tensor: (ids, vals, lse).
    vals are log-probabilities when with_lse, else raw values."""
    lib = _lib.load()
    assert logits.is_cuda and logits.dim() == 2 and logits.stride(1) == 1
    rows, V = logits.shape
    ld = logits.stride(0)
    dev = logits.device
    ids = torch.empty(rows, k, dtype=torch.int32, device=dev)
    vals = torch.empty(rows, k, dtype=torch.float32, device=dev)
    lse = torch.empty(rows, dtype=torch.float32, device=dev) if with_lse else None
    check(lib.eagle_row_topk(_ptr(logits), _dtype_code(logits.dtype), rows, V, ld, k, _ptr(ids),
                             _ptr(vals), _ptr(lse), _stream(dev, stream)), "eagle_row_topk")
    return ids, vals, lse


def expand(level, topk, depth, row_ids, row_logp, front_cand_in, front_S_in, pool, front_out=None,
           stream=None):
    """Stateless expand of one level; pool is a dict of [B][n_cand] tensors (tok, S, parent,
    row) updated in place; front_out = (cand, S) [B][k] tensors or None."""
    lib = _lib.load()
    B = pool["tok"].shape[0]
    fc, fs = (None, None) if front_out is None else front_out
    check(lib.eagle_expand(level, B, topk, depth, _ptr(row_ids), _ptr(row_logp), _ptr(front_cand_in),
                           _ptr(front_S_in), _ptr(fc), _ptr(fs), _ptr(pool["tok"]),
                           _ptr(pool["S"]), _ptr(pool["parent"]), _ptr(pool["row"]),
                           _stream(row_ids.device, stream)), "eagle_expand")


def build_tree(topk, depth, num_keep, pool_tok, pool_S, pool_parent, root_token, pos_base=None,
               status=None, stream=None):
    lib = _lib.load()
    B = pool_tok.shape[0]
    n = num_keep + 1
    W = (n + 31) // 32
    dev = pool_tok.device
    i32 = dict(dtype=torch.int32, device=dev)
    out = {"tokens": torch.empty(B, n, **i32), "parents": torch.empty(B, n, **i32),
           "positions": torch.empty(B, n, **i32), "mask": torch.empty(B, n, W, **i32),
           "logscore": torch.empty(B, n, dtype=torch.float32, device=dev)}
    check(lib.eagle_build_tree(B, topk, depth, num_keep, _ptr(pool_tok), _ptr(pool_S),
                               _ptr(pool_parent), _ptr(root_token), _ptr(pos_base),
                               _ptr(out["tokens"]), _ptr(out["parents"]), _ptr(out["positions"]),
                               _ptr(out["mask"]), _ptr(out["logscore"]), _ptr(status),
                               _stream(dev, stream)), "eagle_build_tree")
    return out


def verify_walk(tokens, parents, target_ids, depth, stream=None):
    lib = _lib.load()
    B, n = tokens.shape
    dev = tokens.device
    i32 = dict(dtype=torch.int32, device=dev)
    out = {"accept_len": torch.empty(B, **i32), "accept_nodes": torch.empty(B, depth + 1, **i32),
           "accept_tokens": torch.empty(B, depth + 1, **i32)}
    check(lib.eagle_verify_walk(B, n, depth, _ptr(tokens), _ptr(parents), _ptr(target_ids),
                                _ptr(out["accept_len"]), _ptr(out["accept_nodes"]),
                                _ptr(out["accept_tokens"]), _stream(dev, stream)),
          "eagle_verify_walk")
    return out


def verify_sample(tokens, parents, target_logits, draft_logits, depth, temperature, u_accept,
                  u_bonus, mode=0, threshold=0.0, scratch=None, stream=None):
    """Sampling tree verification on the GPU (mode 0: recursive rejection sampling, mode 1:
    threshold).  tokens / parents [B][n] int32, logits [B][n][V] fp32, u_accept [B][n] and
    u_bonus [B] fp32 uniforms.  Returns accept_len / accept_nodes / accept_tokens."""
    lib = _lib.load()
    B, n = tokens.shape
    V = target_logits.shape[-1]
    dev = tokens.device
    for t in (target_logits, draft_logits, u_accept, u_bonus):
        assert t.dtype == torch.float32 and t.is_contiguous()
    if scratch is None:
        scratch = torch.empty(B, V, dtype=torch.float32, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    out = {"accept_len": torch.empty(B, **i32), "accept_nodes": torch.empty(B, depth + 1, **i32),
           "accept_tokens": torch.empty(B, depth + 1, **i32)}
    check(lib.eagle_verify_sample(B, n, V, depth, _ptr(tokens), _ptr(parents), _ptr(target_logits),
                                  _ptr(draft_logits), float(temperature), int(mode), float(threshold),
                                  _ptr(u_accept), _ptr(u_bonus), _ptr(scratch),
                                  _ptr(out["accept_len"]), _ptr(out["accept_nodes"]),
                                  _ptr(out["accept_tokens"]), _stream(dev, stream)),
          "eagle_verify_sample")
    return out


def linear_bf16(w, x, bias=None, out_bf16=False, stream=None):
    """Y = X W^T (+ bias) for bf16 W [M][K], X [rows][K] (rows <= 32768, in chunks of 256) on the
    tensor cores."""
    lib = _lib.load()
    M, K = w.shape
    rows = x.shape[0]
    dev = w.device
    y = torch.empty(rows, M, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
    nbytes = lib.eagle_linear_workspace_bytes(M, rows)
    ws = torch.zeros(max(nbytes, 1), dtype=torch.uint8, device=dev)
    check(lib.eagle_linear_bf16(_ptr(w), w.stride(0), _ptr(x), x.stride(0), _ptr(bias), M, K, rows,
                                _ptr(y), y.stride(0), int(out_bf16), _ptr(ws), nbytes,
                                _stream(dev, stream)), "eagle_linear_bf16")
    return y


class DecoderLayer:
    """The draft decoder layer (eagle_decoder_layer): one Llama layer over each request's tree
    nodes with tree attention over a KV cache.  Weights are bf16 CUDA tensors: w_qkv
    [(H + 2 Hkv) D][h], w_o [h][H D], w_norm [h], w_gu [2 I][h], w_d [h][I].  The scratch is
    allocated (zero-filled) on first use and grown as needed."""

    def __init__(self, w_qkv, w_o, w_norm, w_gu, w_d, heads: int, kv_heads: int,
                 rope_theta: float = 10000.0, rms_eps: float = 1e-6):
        self._lib = _lib.load()
        for t, name in ((w_qkv, "w_qkv"), (w_o, "w_o"), (w_norm, "w_norm"), (w_gu, "w_gu"), (w_d, "w_d")):
            _need(t, name, torch.bfloat16)
        h = w_norm.shape[0]
        D = w_qkv.shape[0] // (heads + 2 * kv_heads)
        inter = w_gu.shape[0] // 2
        if w_qkv.shape != (D * (heads + 2 * kv_heads), h) or w_o.shape != (h, heads * D) \
                or w_gu.shape != (2 * inter, h) or w_d.shape != (h, inter):
            raise ValueError("decoder layer weight shapes do not agree")
        self._keep = (w_qkv, w_o, w_norm, w_gu, w_d)
        self.w = _lib.DecoderLayerWeights(h, heads, kv_heads, D, inter, rope_theta, rms_eps,
                                          w_qkv.data_ptr(), w_o.data_ptr(), w_norm.data_ptr(),
                                          w_gu.data_ptr(), w_d.data_ptr())
        self.hidden, self.heads, self.kv_heads, self.head_dim, self.inter = h, heads, kv_heads, D, inter
        self.device = w_qkv.device
        self._ws = None

    def workspace(self, batch: int, nodes: int):
        nbytes = self._lib.eagle_decoder_layer_workspace_bytes(ctypes.byref(self.w), batch, nodes)
        if nbytes == 0:
            raise ValueError(f"unusable decoder layer sizes (batch={batch}, nodes={nodes})")
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        return self._ws, nbytes

    def __call__(self, x, k_cache, v_cache, positions, mask, out=None, new_kv: bool = False, stream=None):
        """x [B][n][h] bf16, k_cache / v_cache [B][P][Hkv][D] bf16 (rotated keys), positions
        [B][n] int32, mask [B][n][ceil(n/32)] int32 ancestor bits.  Returns out [B][n][h] bf16
        (and k_new, v_new [B][n][Hkv][D] if new_kv)."""
        _need(x, "x", torch.bfloat16)
        B, n, h = x.shape
        if h != self.hidden:
            raise ValueError("x hidden size does not match the weights")
        P = 0 if k_cache is None else k_cache.shape[1]
        if P:
            _need(k_cache, "k_cache", torch.bfloat16)
            _need(v_cache, "v_cache", torch.bfloat16)
            if k_cache.shape != (B, P, self.kv_heads, self.head_dim) or v_cache.shape != k_cache.shape:
                raise ValueError("cache shape does not match")
        _need(positions, "positions", torch.int32)
        _need(mask, "mask", torch.int32)
        if positions.shape != (B, n) or mask.shape != (B, n, (n + 31) // 32):
            raise ValueError("positions / mask shape does not match")
        if out is None:
            out = torch.empty_like(x)
        kn = vn = None
        if new_kv:
            kn = torch.empty(B, n, self.kv_heads, self.head_dim, dtype=torch.bfloat16, device=x.device)
            vn = torch.empty_like(kn)
        ws, nbytes = self.workspace(max(B, 1), n)
        check(self._lib.eagle_decoder_layer(ctypes.byref(self.w), B, n, P, _ptr(x),
                                            _ptr(k_cache) if P else None, _ptr(v_cache) if P else None,
                                            _ptr(positions), _ptr(mask), _ptr(out), _ptr(kn), _ptr(vn),
                                            _ptr(ws), nbytes, _stream(x.device, stream)),
              "eagle_decoder_layer")
        return (out, kn, vn) if new_kv else out
