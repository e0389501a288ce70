"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports every entry point
that include/eagle_tree.h declares, and rejects bad arguments on the host before any launch."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "eagle_tree.h"


@pytest.fixture(scope="module")
def lib():
    from eagle_speculative_decoding_draft_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_symbols():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"EAGLE_API\s+[\w\s\*]+?\b(eagle_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("eagle_tree_init", "eagle_draft_level", "eagle_rerank_build_tree",
              "eagle_verify_greedy", "eagle_tree_status", "eagle_tree_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_exports_nothing_else(lib):
    import subprocess
    from eagle_speculative_decoding_draft_gb300._lib import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", str(LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(declared_symbols())


def test_status_strings(lib):
    for code, name in [(0, b"EAGLE_OK"), (1, b"EAGLE_ERR_INVALID_ARG"), (3, b"EAGLE_ERR_STATE"),
                       (5, b"EAGLE_ERR_DEVICE_TIMEOUT"), (6, b"EAGLE_ERR_DEVICE_BOUNDS")]:
        assert lib.eagle_status_str(code) == name


def _cfg(**kw):
    from eagle_speculative_decoding_draft_gb300._lib import TreeConfig
    base = dict(batch=1, hidden=256, vocab=1024, depth=3, topk=2, num_keep=6, dtype=0,
                fc_weight=256, fc_bias=None, lm_head=256, embedding=256)
    base.update(kw)
    return TreeConfig(**base)


@pytest.mark.parametrize("bad", [dict(topk=0), dict(topk=17), dict(depth=0), dict(depth=33),
                                 dict(num_keep=11), dict(num_keep=-1), dict(hidden=250, dtype=1),
                                 dict(hidden=6), dict(batch=-1), dict(vocab=1, topk=2),
                                 dict(dtype=7), dict(depth=30, topk=16)])
def test_init_rejects_bad_configs_on_the_host(lib, bad):
    h = ctypes.c_void_p()
    cfg = _cfg(**bad)
    assert lib.eagle_tree_init(ctypes.byref(cfg), ctypes.c_void_p(4096), 1 << 30, ctypes.byref(h)) == 1
    assert lib.eagle_tree_workspace_bytes(ctypes.byref(cfg)) == 0


def test_init_rejects_null_and_misaligned_pointers(lib):
    h = ctypes.c_void_p()
    cfg = _cfg()
    assert lib.eagle_tree_init(None, ctypes.c_void_p(4096), 1 << 30, ctypes.byref(h)) == 1
    assert lib.eagle_tree_init(ctypes.byref(cfg), None, 1 << 30, ctypes.byref(h)) == 1
    assert lib.eagle_tree_init(ctypes.byref(cfg), ctypes.c_void_p(4096 + 8), 1 << 30,
                               ctypes.byref(h)) == 1
    cfg2 = _cfg(lm_head=None)
    assert lib.eagle_tree_init(ctypes.byref(cfg2), ctypes.c_void_p(4096), 1 << 30,
                               ctypes.byref(h)) == 1
    cfg3 = _cfg(fc_weight=4096 + 4)
    assert lib.eagle_tree_init(ctypes.byref(cfg3), ctypes.c_void_p(4096), 1 << 30,
                               ctypes.byref(h)) == 1


def test_stateless_entries_reject_bad_sizes_on_the_host(lib):
    P = ctypes.c_void_p
    assert lib.eagle_row_topk(P(256), 0, 4, 100, 100, 0, P(256), P(256), None, None) == 1
    assert lib.eagle_row_topk(P(256), 0, 4, 100, 100, 17, P(256), P(256), None, None) == 1
    assert lib.eagle_row_topk(P(256), 0, 4, 100, 99, 2, P(256), P(256), None, None) == 1
    assert lib.eagle_row_topk(P(256), 3, 4, 100, 100, 2, P(256), P(256), None, None) == 1
    assert lib.eagle_row_topk(None, 0, 0, 100, 100, 2, None, None, None, None) == 0  # empty
    assert lib.eagle_expand(3, 1, 2, 3, *([P(256)] * 10), None) == 1  # level >= depth
    assert lib.eagle_expand(0, 0, 2, 3, *([None] * 10), None) == 0    # empty batch
    assert lib.eagle_build_tree(1, 2, 3, 11, *([P(256)] * 11), None) == 1  # m > n_cand
    assert lib.eagle_verify_walk(1, 0, 3, *([P(256)] * 6), None) == 1
    assert lib.eagle_linear_bf16(P(256), 64, P(256), 64, None, 128, 64, 32769, P(256), 128, 0,
                                 P(256), 1 << 20, None) == 1  # rows > 32768
    assert lib.eagle_linear_bf16(P(256), 60, P(256), 64, None, 128, 60, 16, P(256), 128, 0,
                                 P(256), 1 << 20, None) == 1  # ldw not a multiple of 8


def test_verify_sample_rejects_bad_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    ptrs_in = [P(256)] * 4
    ptrs_out = [P(256)] * 6
    ok = lib.eagle_verify_sample
    assert ok(1, 0, 10, 1, *ptrs_in, 1.0, 0, 0.0, *ptrs_out, None) == 1      # no nodes
    assert ok(1, 5000, 10, 1, *ptrs_in, 1.0, 0, 0.0, *ptrs_out, None) == 1   # too many nodes
    assert ok(1, 5, 10, 1, *ptrs_in, 0.0, 0, 0.0, *ptrs_out, None) == 1      # temperature 0
    assert ok(1, 5, 10, 1, *ptrs_in, -1.0, 0, 0.0, *ptrs_out, None) == 1
    assert ok(1, 5, 10, 1, *ptrs_in, float("nan"), 0, 0.0, *ptrs_out, None) == 1
    assert ok(1, 5, 10, 1, *ptrs_in, 1.0, 2, 0.0, *ptrs_out, None) == 1      # mode
    assert ok(1, 5, 10, 1, *ptrs_in, 1.0, 0, 0.0, *([None] + ptrs_out[1:]), None) == 1
    assert ok(0, 5, 10, 1, *([None] * 4), 1.0, 0, 0.0, *([None] * 6), None) == 0  # empty batch


def test_bounded_wait_hook_rejects_bad_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    assert lib.eagle_test_bounded_wait(0, P(256), None) == 1
    assert lib.eagle_test_bounded_wait(-5, P(256), None) == 1
    assert lib.eagle_test_bounded_wait(10**11, P(256), None) == 1
    assert lib.eagle_test_bounded_wait(1000, None, None) == 1


@pytest.mark.parametrize("spec", [[[1, 0]], [[0, 0], [0, 0]], [[0, 0], [1, 0], [0, 1]], [[0, 16]], []])
def test_static_init_rejects_malformed_shapes_on_the_host(lib, spec):
    import numpy as np
    sp = np.ascontiguousarray(np.asarray(spec, dtype=np.int32).reshape(-1, 2))
    cfg = _cfg(depth=2, num_keep=max(1, len(spec)))
    h = ctypes.c_void_p()
    ptr = sp.ctypes.data_as(ctypes.c_void_p)
    assert lib.eagle_tree_workspace_bytes_static(ctypes.byref(cfg), len(spec), ptr) == 0
    assert lib.eagle_tree_init_static(ctypes.byref(cfg), len(spec), ptr, ctypes.c_void_p(4096), 1 << 30,
                                      ctypes.byref(h)) == 1


def test_static_init_checks_depth_and_size_against_the_shape(lib):
    import numpy as np
    sp = np.ascontiguousarray(np.array([[0, 0], [0, 1], [1, 0]], dtype=np.int32))
    ptr = sp.ctypes.data_as(ctypes.c_void_p)
    h = ctypes.c_void_p()
    for cfg in (_cfg(depth=3, num_keep=3), _cfg(depth=2, num_keep=4), _cfg(depth=2, num_keep=3, vocab=1)):
        assert lib.eagle_tree_init_static(ctypes.byref(cfg), 3, ptr, ctypes.c_void_p(4096), 1 << 30,
                                          ctypes.byref(h)) == 1



def test_decoder_layer_rejects_bad_arguments_on_the_host(lib):
    from eagle_speculative_decoding_draft_gb300._lib import DecoderLayerWeights
    P = ctypes.c_void_p

    def weights(**kw):
        f = dict(hidden=256, heads=4, kv_heads=2, head_dim=64, inter=512, rope_theta=1e4, rms_eps=1e-6,
                 w_qkv=256, w_o=256, w_norm=256, w_gu=256, w_d=256)
        f.update(kw)
        return DecoderLayerWeights(*(f[k] for k, _ in DecoderLayerWeights._fields_))

    def call(w, batch=2, nodes=9, prefix=5, x=P(256), kc=P(256), vc=P(256), kn=None, vn=None, ws=P(256)):
        return lib.eagle_decoder_layer(ctypes.byref(w), batch, nodes, prefix, x, kc, vc, P(256), P(256), P(256),
                                       kn, vn, ws, 1 << 30, None)

    good = weights()
    for bad in (weights(head_dim=48), weights(head_dim=256), weights(heads=3), weights(hidden=252),
                weights(inter=100), weights(rope_theta=0.0), weights(rms_eps=-1.0), weights(w_o=0),
                weights(w_gu=264)):
        assert call(bad) == 1
        assert lib.eagle_decoder_layer_workspace_bytes(ctypes.byref(bad), 2, 9) == 0
    assert call(good, nodes=0) == 1
    assert call(good, nodes=4098) == 1
    assert call(good, prefix=-1) == 1
    assert call(good, x=P(264)) == 1                 # x not 16-byte aligned
    assert call(good, kc=None) == 1                  # a cache is needed when prefix > 0
    assert call(good, kn=P(256)) == 1                # k_new without v_new
    assert call(good, ws=P(128)) == 1                # workspace not 256-byte aligned
    assert call(good, batch=0, x=None, kc=None, vc=None, ws=None) == 0  # empty batch
    assert lib.eagle_decoder_layer_workspace_bytes(ctypes.byref(good), 2, 0) == 0
