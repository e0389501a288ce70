"""CPU oracle of one EAGLE / EAGLE-2 dynamic draft-tree step (ctypes shim over plain C).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The CUDA library never loads it and shares no
code with it; the product path fails loudly when its own extension is missing instead of
falling back here.

The arithmetic lives in ``eagle_oracle.c`` (plain loops, fp32 accumulation in ascending index
order, ties to the lowest index).  This module only compiles that file with gcc when the shared
object is missing or stale, and marshals numpy arrays in and out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "eagle_oracle.c"
_LIB = _HERE / "liboracle.so"
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_ERR_ARG, ORC_ERR_TREE, ORC_ERR_NOMEM = 0, 1, 2, 3


def build(force: bool = False) -> Path:
    """Compile the oracle with gcc (OpenMP over output elements, no FMA contraction)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", str(tmp), str(_SRC), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("hidden", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("depth", ctypes.c_int32), ("topk", ctypes.c_int32), ("num_keep", ctypes.c_int32),
                ("is_bf16", ctypes.c_int32)]


class LayerDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("nodes", ctypes.c_int32), ("prefix", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("inter", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("rms_eps", ctypes.c_float)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(str(_LIB))
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            L.orc_bf16_to_f32.restype = ctypes.c_float
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f32_to_bf16.restype = ctypes.c_uint16
            L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            L.orc_round_bf16_array.restype = None
            L.orc_round_bf16_array.argtypes = [ctypes.c_int64, P, P]
            L.orc_num_threads.restype = i32
            L.orc_set_num_threads.argtypes = [i32]
            L.orc_fc_row.restype = None
            L.orc_fc_row.argtypes = [i32, i32, P, P, P, P, i32, P]
            L.orc_lm_head_row.restype = None
            L.orc_lm_head_row.argtypes = [i32, i32, i32, P, P, P]
            L.orc_log_softmax_topk.restype = None
            L.orc_log_softmax_topk.argtypes = [i32, i32, P, P, P, P]
            L.orc_num_candidates.restype = i32
            L.orc_num_candidates.argtypes = [i32, i32]
            L.orc_draft_tree.restype = i32
            L.orc_draft_tree.argtypes = [ctypes.POINTER(Dims)] + [P] * 24
            L.orc_verify_greedy.restype = i32
            L.orc_verify_greedy.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P]
            L.orc_decoder_layer.restype = i32
            L.orc_decoder_layer.argtypes = [ctypes.POINTER(LayerDims)] + [P] * 13
            L.orc_draft_static.restype = i32
            L.orc_draft_static.argtypes = [ctypes.POINTER(Dims)] + [P] * 7 + [i32] + [P] * 7
            L.orc_draft_extend.restype = i32
            L.orc_draft_extend.argtypes = [ctypes.POINTER(Dims)] + [P] * 5 + [i32] + [P] * 10
            L.orc_verify_sample.restype = i32
            L.orc_verify_sample.argtypes = [i32, i32, i32, i32, P, P, P, P, ctypes.c_double, i32,
                                            ctypes.c_double, P, P, P, P, P]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def raw(t, is_bf16: bool):
    """A C-contiguous numpy array of the raw element bits: uint16 for bf16, float32 otherwise.

    Accepts numpy arrays or torch tensors (bf16 tensors are viewed as their bit patterns)."""
    if t is None:
        return None
    if hasattr(t, "detach"):  # torch tensor
        import torch
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return np.ascontiguousarray(t.numpy())
    a = np.ascontiguousarray(t)
    if is_bf16 and a.dtype != np.uint16:
        raise TypeError("bf16 data must be given as uint16 bit patterns")
    if not is_bf16 and a.dtype != np.float32:
        raise TypeError("fp32 data must be float32")
    return a


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


def num_candidates(depth: int, k: int) -> int:
    return int(lib().orc_num_candidates(depth, k))


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32: the upper half of a binary32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (the oracle's own rounding)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_round_bf16_array(x.size, _ptr(x), _ptr(out))
    return out


def fc_row(w_fc, b_fc, feat, emb, tok: int, is_bf16: bool) -> np.ndarray:
    """f^ = round(W_fc [feat || E[tok]] + b): one draft FC row (fp32 array of length h)."""
    w = raw(w_fc, is_bf16)
    b = raw(b_fc, is_bf16)
    e = raw(emb, is_bf16)
    f = np.ascontiguousarray(feat, dtype=np.float32)
    h = w.shape[0]
    out = np.empty(h, dtype=np.float32)
    lib().orc_fc_row(h, int(is_bf16), _ptr(w), _ptr(b), _ptr(f), _ptr(e), int(tok), _ptr(out))
    return out


def lm_head_row(w_lm, fhat, is_bf16: bool) -> np.ndarray:
    """z = W_lm f^ (fp32 array of length V)."""
    w = raw(w_lm, is_bf16)
    f = np.ascontiguousarray(fhat, dtype=np.float32)
    V, h = w.shape
    out = np.empty(V, dtype=np.float32)
    lib().orc_lm_head_row(h, V, int(is_bf16), _ptr(w), _ptr(f), _ptr(out))
    return out


def log_softmax_topk(z, k: int):
    """(ids[k] int32, logp[k] float32, lse float) of one logit row."""
    z = np.ascontiguousarray(z, dtype=np.float32)
    ids = np.empty(k, dtype=np.int32)
    logp = np.empty(k, dtype=np.float32)
    lse = np.empty(1, dtype=np.float32)
    lib().orc_log_softmax_topk(z.shape[0], k, _ptr(z), _ptr(ids), _ptr(logp), _ptr(lse))
    return ids, logp, float(lse[0])


def draft_tree(w_fc, b_fc, w_lm, emb, root_feat, root_tok, depth: int, topk: int, num_keep: int,
               is_bf16: bool, pos_base=None, rows: bool = True, row_logits: bool = False,
               node_logits: bool = False) -> dict:
    """Run one draft-tree step for a batch; returns every intermediate as numpy arrays.

    Keys: row_fhat [d][R][h], row_z [d][R][V] (if row_logits), row_lse [d][R],
    row_ids / row_logp [d][R][k], front_cand [d][B][k], cand_tok / cand_S / cand_parent /
    cand_row [B][n_cand], tree_tok / tree_parent / tree_pos / tree_S / tree_cand [B][m+1],
    tree_mask [B][m+1][W] (uint32), node_z [B][m+1][V] (if node_logits).  R = B*k."""
    w1, b1, w2, e = (raw(w_fc, is_bf16), raw(b_fc, is_bf16), raw(w_lm, is_bf16),
                     raw(emb, is_bf16))
    f = raw(root_feat, is_bf16)
    rt = np.ascontiguousarray(root_tok, dtype=np.int32)
    pb = None if pos_base is None else np.ascontiguousarray(pos_base, dtype=np.int32)
    h = w1.shape[0]
    V = w2.shape[0]
    B = rt.shape[0]
    d, k, m = depth, topk, num_keep
    R = B * k
    nc = num_candidates(d, k)
    n = m + 1
    W = (n + 31) // 32
    out = {}
    z32 = np.float32
    if rows:
        out["row_fhat"] = np.zeros((d, R, h), z32)
        out["row_lse"] = np.zeros((d, R), z32)
        out["row_ids"] = np.full((d, R, k), -1, np.int32)
        out["row_logp"] = np.zeros((d, R, k), z32)
    if row_logits:
        out["row_z"] = np.zeros((d, R, V), z32)
    out["front_cand"] = np.full((d, B, k), -1, np.int32)
    out["cand_tok"] = np.zeros((B, nc), np.int32)
    out["cand_S"] = np.zeros((B, nc), z32)
    out["cand_parent"] = np.zeros((B, nc), np.int32)
    out["cand_row"] = np.zeros((B, nc), np.int32)
    out["tree_tok"] = np.zeros((B, n), np.int32)
    out["tree_parent"] = np.zeros((B, n), np.int32)
    out["tree_pos"] = np.zeros((B, n), np.int32)
    out["tree_mask"] = np.zeros((B, n, W), np.uint32)
    out["tree_S"] = np.zeros((B, n), z32)
    out["tree_cand"] = np.zeros((B, n), np.int32)
    if node_logits:
        out["node_z"] = np.zeros((B, n, V), z32)
    dims = Dims(B, h, V, d, k, m, int(is_bf16))
    g = out.get
    rc = lib().orc_draft_tree(
        ctypes.byref(dims), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(e), _ptr(f), _ptr(rt), _ptr(pb),
        _ptr(g("row_fhat")), _ptr(g("row_z")), _ptr(g("row_lse")), _ptr(g("row_ids")),
        _ptr(g("row_logp")), _ptr(out["front_cand"]), _ptr(out["cand_tok"]),
        _ptr(out["cand_S"]), _ptr(out["cand_parent"]), _ptr(out["cand_row"]),
        _ptr(out["tree_tok"]), _ptr(out["tree_parent"]), _ptr(out["tree_pos"]),
        _ptr(out["tree_mask"]), _ptr(out["tree_S"]), _ptr(out["tree_cand"]),
        _ptr(g("node_z")))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_draft_tree failed with code {rc}")
    return out


def decoder_layer(x, w_qkv, w_o, w_norm, w_gu, w_d, k_cache, v_cache, pos, mask, heads: int,
                  kv_heads: int, rope_theta: float = 10000.0, rms_eps: float = 1e-6,
                  new_kv: bool = False) -> dict:
    """One draft decoder layer over each request's tree (see orc_decoder_layer).  Tensors are bf16
    (torch) except pos [B][n] int32 and mask [B][n][W] (int32/uint32).  x [B][n][h], k_cache /
    v_cache [B][P][Hkv][D].  Returns out [B][n][h] as float32 (bf16 values) and, if new_kv, the
    tree's rotated keys and values [B][n][Hkv][D]."""
    X = raw(x, True)
    B, n, h = X.shape
    KC = raw(k_cache, True)
    P, D = KC.shape[1], KC.shape[3]
    wgu = raw(w_gu, True)
    I = wgu.shape[0] // 2
    dims = LayerDims(B, n, P, h, heads, kv_heads, D, I, rope_theta, rms_eps)
    out = np.zeros((B, n, h), np.uint16)
    kn = np.zeros((B, n, kv_heads, D), np.uint16) if new_kv else None
    vn = np.zeros((B, n, kv_heads, D), np.uint16) if new_kv else None
    pz = np.ascontiguousarray(pos, dtype=np.int32)
    mz = np.ascontiguousarray(np.asarray(mask).view(np.uint32) if np.asarray(mask).dtype == np.int32
                              else np.asarray(mask, dtype=np.uint32))
    rc = lib().orc_decoder_layer(ctypes.byref(dims), _ptr(X), _ptr(raw(w_qkv, True)), _ptr(raw(w_o, True)),
                                 _ptr(raw(w_norm, True)), _ptr(wgu), _ptr(raw(w_d, True)), _ptr(KC),
                                 _ptr(raw(v_cache, True)), _ptr(pz), _ptr(mz), _ptr(out), _ptr(kn), _ptr(vn))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_decoder_layer failed with code {rc}")
    f = lambda a: (a.astype(np.uint32) << 16).view(np.float32)
    res = {"out": f(out)}
    if new_kv:
        res["k_new"], res["v_new"] = f(kn), f(vn)
    return res


def draft_static(w_fc, b_fc, w_lm, emb, root_feat, root_tok, spec, is_bf16: bool, pos_base=None,
                 node_fhat: bool = False) -> dict:
    """EAGLE-1 static tree (see orc_draft_static).  spec: [N][2] (parent, rank) for drafted
    nodes 1..N.  Returns tree_tok / tree_parent / tree_pos / tree_S [B][N+1], tree_mask
    [B][N+1][W] (uint32) and node_fhat [B][N+1][h] (if asked)."""
    w1, b1, w2, e = (raw(w_fc, is_bf16), raw(b_fc, is_bf16), raw(w_lm, is_bf16), raw(emb, is_bf16))
    f = raw(root_feat, is_bf16)
    rt = np.ascontiguousarray(root_tok, dtype=np.int32)
    pb = None if pos_base is None else np.ascontiguousarray(pos_base, dtype=np.int32)
    sp = np.ascontiguousarray(np.asarray(spec, dtype=np.int32).reshape(-1, 2))
    h, V, B, N = w1.shape[0], w2.shape[0], rt.shape[0], sp.shape[0]
    n = N + 1
    W = (n + 31) // 32
    out = {"tree_tok": np.zeros((B, n), np.int32), "tree_parent": np.zeros((B, n), np.int32),
           "tree_pos": np.zeros((B, n), np.int32), "tree_mask": np.zeros((B, n, W), np.uint32),
           "tree_S": np.zeros((B, n), np.float32),
           "node_fhat": np.zeros((B, n, h), np.float32) if node_fhat else None}
    dims = Dims(B, h, V, 1, 1, N, int(is_bf16))
    rc = lib().orc_draft_static(ctypes.byref(dims), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(e), _ptr(f), _ptr(rt),
                                _ptr(pb), N, _ptr(sp), _ptr(out["tree_tok"]), _ptr(out["tree_parent"]),
                                _ptr(out["tree_pos"]), _ptr(out["tree_mask"]), _ptr(out["tree_S"]),
                                _ptr(out["node_fhat"]))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_draft_static failed with code {rc}")
    return out


def draft_extend(w_fc, b_fc, w_lm, emb, node_feat, accept_len, accept_nodes, accept_tok,
                 depth: int, topk: int, is_bf16: bool, logits: bool = True) -> dict:
    """Draft extend over each request's accepted path (see orc_draft_extend).  node_feat
    [B][n][h] (torch bf16 or fp32 tensor, or numpy fp32); accept_* from the verify.  Returns
    next_feat [B][h] fp32, next_tok [B], path_fhat [B][d+1][h], path_z [B][d+1][V] (if logits),
    ids / logp [B][k] and lse [B] of the last verified row."""
    fc, bfc, lm, em = (raw(w_fc, is_bf16), raw(b_fc, is_bf16), raw(w_lm, is_bf16), raw(emb, is_bf16))
    if hasattr(node_feat, "detach"):  # torch: widen bf16 exactly
        F = np.ascontiguousarray(node_feat.detach().cpu().float().numpy())
    else:
        F = np.ascontiguousarray(node_feat, dtype=np.float32)
    B, n, h = F.shape
    V = lm.shape[0]
    al = np.ascontiguousarray(accept_len, dtype=np.int32)
    an = np.ascontiguousarray(accept_nodes, dtype=np.int32)
    at = np.ascontiguousarray(accept_tok, dtype=np.int32)
    dims = Dims(B, h, V, depth, topk, 0, int(is_bf16))
    out = {"next_feat": np.zeros((B, h), np.float32), "next_tok": np.zeros(B, np.int32),
           "path_fhat": np.zeros((B, depth + 1, h), np.float32),
           "path_z": np.zeros((B, depth + 1, V), np.float32) if logits else None,
           "ids": np.zeros((B, topk), np.int32), "logp": np.zeros((B, topk), np.float32),
           "lse": np.zeros(B, np.float32)}
    rc = lib().orc_draft_extend(ctypes.byref(dims), _ptr(fc), _ptr(bfc), _ptr(lm), _ptr(em), _ptr(F), n,
                                _ptr(al), _ptr(an), _ptr(at), _ptr(out["next_feat"]),
                                _ptr(out["next_tok"]), _ptr(out["path_fhat"]), _ptr(out["path_z"]),
                                _ptr(out["ids"]), _ptr(out["logp"]), _ptr(out["lse"]))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_draft_extend failed with code {rc}")
    return out


def verify_sample(tree_tok, tree_parent, target, draft, depth: int, temperature: float,
                  u_acc, u_bonus, mode: int = 0, threshold: float = 0.0) -> dict:
    """Sampling tree verification (mode 0: recursive rejection sampling; mode 1: threshold).
    target, draft: [B][n][V] float32 logits; u_acc [B][n], u_bonus [B] uniforms in [0, 1).
    Returns accept_len [B] and accept_nodes / accept_tok [B][depth+1] (bonus last)."""
    tt = np.ascontiguousarray(tree_tok, dtype=np.int32)
    tp = np.ascontiguousarray(tree_parent, dtype=np.int32)
    T = np.ascontiguousarray(target, dtype=np.float32)
    Z = np.ascontiguousarray(draft, dtype=np.float32)
    ua = np.ascontiguousarray(u_acc, dtype=np.float32)
    ub = np.ascontiguousarray(u_bonus, dtype=np.float32)
    B, n = tt.shape
    V = T.shape[-1]
    assert T.shape == (B, n, V) and Z.shape == (B, n, V) and ua.shape == (B, n) and ub.shape == (B,)
    al = np.zeros(B, np.int32)
    an = np.zeros((B, depth + 1), np.int32)
    at = np.zeros((B, depth + 1), np.int32)
    rc = lib().orc_verify_sample(B, n, V, depth, _ptr(tt), _ptr(tp), _ptr(T), _ptr(Z),
                                 float(temperature), int(mode), float(threshold), _ptr(ua),
                                 _ptr(ub), _ptr(al), _ptr(an), _ptr(at))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_verify_sample failed with code {rc}")
    return {"accept_len": al, "accept_nodes": an, "accept_tok": at}


def verify_greedy(tree_tok, tree_parent, target, depth: int) -> dict:
    """Greedy tree verification. target: [B][n][V] float32.  Returns accept_len [B],
    accept_nodes / accept_tok [B][depth+1] and g [B][n] (the target argmax per node)."""
    tt = np.ascontiguousarray(tree_tok, dtype=np.int32)
    tp = np.ascontiguousarray(tree_parent, dtype=np.int32)
    T = np.ascontiguousarray(target, dtype=np.float32)
    B, n = tt.shape
    V = T.shape[-1]
    assert T.shape == (B, n, V)
    g = np.zeros((B, n), np.int32)
    al = np.zeros(B, np.int32)
    an = np.zeros((B, depth + 1), np.int32)
    at = np.zeros((B, depth + 1), np.int32)
    rc = lib().orc_verify_greedy(B, n, V, depth, _ptr(tt), _ptr(tp), _ptr(T), _ptr(g), _ptr(al),
                                 _ptr(an), _ptr(at))
    if rc != ORC_OK:
        raise RuntimeError(f"orc_verify_greedy failed with code {rc}")
    return {"accept_len": al, "accept_nodes": an, "accept_tok": at, "g": g}
