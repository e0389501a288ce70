"""EAGLE-1 static draft trees on the GPU (eagle_tree_init_static).

fp32 shapes against the oracle (structure and tokens exact, scores within 1e-4); bf16 shapes
against the oracle (structure exact; a node's ranked token may differ only where the oracle's
logits of its parent's row leave a margin of at most max(1e-3, twice the GPU-oracle deviation of
that row); where none differs, tokens exact and scores and node logits within 2e-2); bf16 static
chains and stars against the GPU's own dynamic trees with topk = 1 and with depth 1 (same rows,
same kernels: bit for bit); a static handle through verify, draft extend and the host step.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_draft_gb300 import synth
from parity import to_np

pytestmark = pytest.mark.gpu

SPARSE = [[0, 0], [0, 1], [0, 2], [1, 0], [1, 1], [2, 0], [3, 0], [3, 1], [4, 0], [5, 0], [7, 0], [7, 3]]
BINARY = [[0, 0], [0, 1], [1, 0], [1, 1], [2, 0], [2, 1]]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    return torch.device("cuda", 0)


def depth_of(spec):
    dep = [0]
    for p, _ in spec:
        dep.append(dep[p] + 1)
    return max(dep)


def handle(dev, w, inp, spec=None, depth=None, topk=None, keep=None):
    from eagle_speculative_decoding_draft_gb300.engine import EagleTree
    g = lambda t: t.to(dev).contiguous()
    return EagleTree(g(inp.w_fc), g(inp.b_fc) if w.bias else None, g(inp.w_lm), g(inp.emb), w.batch,
                     depth if depth is not None else depth_of(spec), topk if topk is not None else 1,
                     keep if keep is not None else len(spec), static_spec=spec)


@pytest.mark.parametrize("spec", [SPARSE, BINARY, [[j, 0] for j in range(5)]], ids=["sparse", "binary", "chain"])
def test_fp32_static_tree_matches_the_oracle(dev, spec):
    w = synth.custom(256, 1500, 3, 1, 1, 1, dtype="fp32")
    inp = synth.make_inputs(w, seed=9)
    eng = handle(dev, w, inp, spec)
    g = lambda t: t.to(dev).contiguous()
    pos = torch.arange(w.batch, dtype=torch.int32) * 11
    eng.draft(g(inp.root_feat), g(inp.root_tok), g(pos))
    tree = {k: to_np(v) for k, v in eng.rerank_build_tree(g(pos)).items()}
    torch.cuda.synchronize()
    ref = oracle.draft_static(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok, spec, False,
                              pos_base=pos.numpy())
    assert np.array_equal(tree["tokens"], ref["tree_tok"])
    assert np.array_equal(tree["parents"], ref["tree_parent"])
    assert np.array_equal(tree["positions"], ref["tree_pos"])
    assert np.array_equal(tree["mask"].view(np.uint32), ref["tree_mask"])
    assert np.max(np.abs(tree["logscore"] - ref["tree_S"])) <= 1e-4
    eng.close()


@pytest.mark.parametrize("spec,h,V", [(SPARSE, 256, 4000), (BINARY, 512, 3000), ([[j, 0] for j in range(6)], 1024, 5000)],
                         ids=["sparse", "binary", "chain"])
def test_bf16_static_tree_matches_the_oracle(dev, spec, h, V):
    from parity import BF16_ABS, MARGIN, assert_close_logits, top_gaps
    w = synth.custom(h, V, 4, 1, 1, 1, dtype="bf16")
    inp = synth.make_inputs(w, seed=h + V)
    eng = handle(dev, w, inp, spec)
    g = lambda t: t.to(dev).contiguous()
    pos = torch.arange(w.batch, dtype=torch.int32) * 5 + 2
    f = g(inp.root_feat)
    tree = {k: to_np(v) for k, v in eng.draft(f, g(inp.root_tok), g(pos)).items()}
    nz = to_np(eng.node_logits(f))
    torch.cuda.synchronize()
    ref = oracle.draft_static(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok, spec, True,
                              pos_base=pos.numpy(), node_fhat=True)
    assert np.array_equal(tree["parents"], ref["tree_parent"])
    assert np.array_equal(tree["positions"], ref["tree_pos"])
    assert np.array_equal(tree["mask"].view(np.uint32), ref["tree_mask"])
    n = len(spec) + 1
    kids = {}
    for j, (p, r) in enumerate(spec, start=1):
        kids.setdefault(p, []).append((j, r))
    exact = 0
    for b in range(w.batch):
        same = True
        for p, ch in sorted(kids.items()):
            # parents come first: every node up to p drafted the oracle's token (else we stopped)
            zo = oracle.lm_head_row(inp.w_lm, ref["node_fhat"][b, p], True)
            dev_z = float(np.max(np.abs(nz[b, p].astype(np.float64) - zo)))
            assert dev_z <= BF16_ABS, f"request {b} node {p}: logits off by {dev_z}"
            want = max(r for _, r in ch) + 2
            mg = float(np.min(top_gaps(zo, want)))
            for j, r in ch:
                if tree["tokens"][b, j] != ref["tree_tok"][b, j]:
                    assert mg <= max(MARGIN, 2 * dev_z), (f"request {b} node {j}: token differs with margin "
                                                         f"{mg:.3g}")
                    same = False
            if not same:
                break
        if same:
            exact += 1
            assert np.all(np.abs(tree["logscore"][b] - ref["tree_S"][b]) <= BF16_ABS)
    assert exact >= 2, f"only {exact} of {w.batch} requests drafted the oracle's tokens"
    eng.close()


def test_bf16_static_chain_and_star_equal_the_dynamic_trees(dev):
    w = synth.WORKLOADS[2]
    inp = synth.make_inputs(w)
    g = lambda t: t.to(dev).contiguous()
    f, t0 = g(inp.root_feat), g(inp.root_tok)
    cases = [([[j, 0] for j in range(6)], dict(depth=6, topk=1, keep=6)),
             ([[0, r] for r in range(10)], dict(depth=1, topk=10, keep=10))]
    for spec, dyn in cases:
        st = handle(dev, w, inp, spec)
        dy = handle(dev, w, inp, None, **dyn)
        a = st.draft(f, t0)
        b = dy.draft(f, t0)
        torch.cuda.synchronize()
        for key in ("tokens", "parents", "positions", "mask", "logscore"):
            assert torch.equal(a[key], b[key]), key
        # node logits follow the same rows
        assert torch.equal(st.node_logits(f), dy.node_logits(f))
        st.close()
        dy.close()


def test_static_handle_through_verify_extend_and_the_host_step(dev):
    w = synth.custom(128, 2000, 4, 1, 1, 1, dtype="bf16")
    inp = synth.make_inputs(w, seed=12)
    eng = handle(dev, w, inp, SPARSE)
    g = lambda t: t.to(dev).contiguous()
    B, n, d = w.batch, len(SPARSE) + 1, depth_of(SPARSE)
    f, t0 = g(inp.root_feat), g(inp.root_tok)
    tree = eng.draft(f, t0)
    nz = eng.node_logits(f)
    T = (nz + 0.3 * torch.randn(nz.shape, device=dev, generator=torch.Generator(device=dev).manual_seed(1))).contiguous()
    ver = eng.verify_greedy(tree["tokens"], tree["parents"], T)
    torch.cuda.synchronize()
    ref = oracle.verify_greedy(to_np(tree["tokens"]), to_np(tree["parents"]), to_np(T), d)
    assert np.array_equal(to_np(ver["accept_len"]), ref["accept_len"])
    assert np.array_equal(to_np(ver["accept_tokens"]), ref["accept_tok"])
    # extend: the next static tree from the returned root equals a fresh one
    F = g(torch.randn(B, n, w.hidden).to(torch.bfloat16))
    nf, nt = eng.extend(F, ver["accept_len"], ver["accept_nodes"], ver["accept_tokens"])
    for lvl in range(1, d):
        eng.draft_level(lvl)
    t1 = eng.rerank_build_tree()
    fresh = handle(dev, w, inp, SPARSE)
    t2 = fresh.draft(nf.contiguous(), nt)
    torch.cuda.synchronize()
    for key in ("tokens", "parents", "positions", "mask", "logscore"):
        assert torch.equal(t1[key], t2[key]), key
    # host step
    i32 = dict(dtype=torch.int32, pin_memory=True)
    host = {"tokens": torch.empty(B, n, **i32), "parents": torch.empty(B, n, **i32),
            "positions": torch.empty(B, n, **i32), "mask": torch.empty(B, n, 1, **i32),
            "accept_len": torch.empty(B, **i32), "accept_tokens": torch.empty(B, d + 1, **i32)}
    staging = torch.empty_like(T)
    eng.step_host(inp.root_feat.pin_memory(), inp.root_tok.pin_memory(), T.cpu().pin_memory(), staging, host)
    assert torch.equal(host["tokens"], tree["tokens"].cpu())
    assert torch.equal(host["accept_len"], ver["accept_len"].cpu())
    eng.status()
    eng.close()
    fresh.close()
