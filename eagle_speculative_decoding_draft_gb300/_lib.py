"""ctypes declarations of the C ABI in include/eagle_tree.h.

Loads the in-tree ``lib/libeagle_tree.so`` and nothing else: when it is missing the import of
any entry point raises, there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import POINTER, c_int, c_int32, c_int64, c_size_t, c_void_p
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "lib" / "libeagle_tree.so"

EAGLE_F32, EAGLE_BF16 = 0, 1
STATUS_NAMES = {
    0: "EAGLE_OK",
    1: "EAGLE_ERR_INVALID_ARG",
    2: "EAGLE_ERR_UNSUPPORTED",
    3: "EAGLE_ERR_STATE",
    4: "EAGLE_ERR_CUDA",
    5: "EAGLE_ERR_DEVICE_TIMEOUT",
    6: "EAGLE_ERR_DEVICE_BOUNDS",
}


class EagleError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


class TreeConfig(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("hidden", c_int32), ("vocab", c_int32), ("depth", c_int32),
                ("topk", c_int32), ("num_keep", c_int32), ("dtype", c_int),
                ("fc_weight", c_void_p), ("fc_bias", c_void_p), ("lm_head", c_void_p),
                ("embedding", c_void_p)]


class TreeLayout(ctypes.Structure):
    _fields_ = [(n, c_int64) for n in ("x", "fhat", "logits", "row_ids", "row_logp", "row_lse",
                                       "pool_tok", "pool_S", "pool_parent", "pool_row",
                                       "front_cand", "front_S", "node_tok", "node_src",
                                       "target_ids", "status")] + \
               [(n, c_int32) for n in ("r_pad", "n_cand", "num_nodes", "mask_words",
                                       "front_current", "num_sms")]


class DecoderLayerWeights(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in ("hidden", "heads", "kv_heads", "head_dim", "inter")] + \
               [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)] + \
               [(n, c_void_p) for n in ("w_qkv", "w_o", "w_norm", "w_gu", "w_d")]


_SIGS = {
    "eagle_tree_workspace_bytes": (c_size_t, [POINTER(TreeConfig)]),
    "eagle_tree_init": (c_int, [POINTER(TreeConfig), c_void_p, c_size_t, POINTER(c_void_p)]),
    "eagle_draft_level": (c_int, [c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "eagle_rerank_build_tree": (c_int, [c_void_p] + [c_void_p] * 6 + [c_void_p]),
    "eagle_verify_greedy": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p]),
    "eagle_tree_node_logits": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p]),
    "eagle_tree_step_host": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p]),
    "eagle_tree_status": (c_int, [c_void_p, c_void_p]),
    "eagle_tree_destroy": (None, [c_void_p]),
    "eagle_status_str": (ctypes.c_char_p, [c_int]),
    "eagle_tree_get_layout": (c_int, [c_void_p, POINTER(TreeLayout)]),
    "eagle_row_topk": (c_int, [c_void_p, c_int, c_int32, c_int32, c_int64, c_int32, c_void_p,
                               c_void_p, c_void_p, c_void_p]),
    "eagle_expand": (c_int, [c_int32, c_int32, c_int32, c_int32] + [c_void_p] * 10 + [c_void_p]),
    "eagle_build_tree": (c_int, [c_int32, c_int32, c_int32, c_int32] + [c_void_p] * 11
                         + [c_void_p]),
    "eagle_verify_walk": (c_int, [c_int32, c_int32, c_int32] + [c_void_p] * 6 + [c_void_p]),
    "eagle_verify_sample": (c_int, [c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                    c_void_p, ctypes.c_float, c_int32, ctypes.c_float, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "eagle_tree_profile": (c_int, [c_void_p, c_int32]),
    "eagle_tree_profile_enable": (c_int, [c_void_p, c_int32]),
    "eagle_tree_profile_read": (c_int, [c_void_p, POINTER(c_int32), POINTER(ctypes.c_double),
                                        POINTER(ctypes.c_double)]),
    "eagle_tree_profile_list": (c_int, [c_void_p, c_int32, POINTER(c_int32), POINTER(ctypes.c_float),
                                        POINTER(ctypes.c_double), POINTER(ctypes.c_double),
                                        POINTER(c_int32)]),
    "eagle_tree_launch_count": (c_int64, [c_void_p]),
    "eagle_tree_step_graphed": (c_int32, [c_void_p]),
    "eagle_draft_extend": (c_int, [c_void_p] * 10),
    "eagle_tree_workspace_bytes_static": (c_size_t, [POINTER(TreeConfig), c_int32, c_void_p]),
    "eagle_tree_init_static": (c_int, [POINTER(TreeConfig), c_int32, c_void_p, c_void_p, c_size_t,
                                       POINTER(c_void_p)]),
    "eagle_test_bounded_wait": (c_int, [c_int64, c_void_p, c_void_p]),
    "eagle_linear_workspace_bytes": (c_size_t, [c_int32, c_int32]),
    "eagle_decoder_layer_workspace_bytes": (c_size_t, [POINTER(DecoderLayerWeights), c_int32, c_int32]),
    "eagle_decoder_layer": (c_int, [POINTER(DecoderLayerWeights), c_int32, c_int32, c_int32]
                            + [c_void_p] * 9 + [c_size_t, c_void_p]),
    "eagle_linear_noalloc_scratch_bytes": (c_size_t, []),
    "eagle_linear_bf16_noalloc": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int32,
                                          c_int32, c_int32, c_void_p, c_int64, c_int32, c_void_p]),
    "eagle_linear_bf16": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int32,
                                  c_int32, c_int32, c_void_p, c_int64, c_int32, c_void_p,
                                  c_size_t, c_void_p]),
}

_lock = threading.Lock()
_lib = None


def load(path: Path | None = None):
    """The loaded CUDA library with typed entry points.  Raises if it has not been built.

    The environment variable EAGLE_TREE_LIB, when set, names another build of the same library
    to load instead (the tests use it for the checking build)."""
    global _lib
    with _lock:
        if _lib is None:
            override = os.environ.get("EAGLE_TREE_LIB")
            p = Path(path) if path else (Path(override) if override else LIB_PATH)
            if not p.exists():
                raise RuntimeError(
                    f"{p} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(str(p))
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def check(code: int, where: str) -> None:
    if code != 0:
        raise EagleError(code, where)
