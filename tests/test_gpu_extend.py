"""Draft extend on the GPU (eagle_draft_extend).

* Closed loop: verify -> extend -> levels 1..d-1 -> rerank/build gives, bit for bit, the tree that
  a fresh handle drafts from the root extend returns (the last verified position's target
  feature and the bonus token): the extend's last row is the next round's level 0.
* Against the oracle: the path rows' FC output within the bf16 rounding of the oracle's, the
  level-0 logits within the logit tolerance, the next root exact.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_draft_gb300 import synth
from parity import BF16_ABS, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    return torch.device("cuda", 0)


def make(dev, w):
    from eagle_speculative_decoding_draft_gb300.engine import EagleTree
    inp = synth.make_inputs(w)
    g = lambda t: t.to(dev).contiguous()
    eng = EagleTree(g(inp.w_fc), g(inp.b_fc) if w.bias else None, g(inp.w_lm), g(inp.emb),
                    w.batch, w.depth, w.topk, w.num_keep)
    return inp, eng


CASES = [synth.WORKLOADS[1], synth.WORKLOADS[2], synth.custom(64, 300, 3, 4, 3, 9, dtype="bf16"),
         synth.custom(128, 1000, 5, 1, 4, 4, dtype="bf16")]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_closed_loop_matches_a_fresh_draft(dev, w):
    inp, eng = make(dev, w)
    _, fresh = make(dev, w)
    g = lambda t: t.to(dev).contiguous()
    B, n, d, h = w.batch, w.num_nodes, w.depth, w.hidden
    fdt = torch.bfloat16 if w.is_bf16 else torch.float32
    rng = np.random.default_rng(17)
    feat, tok = g(inp.root_feat), g(inp.root_tok)
    for rnd in range(3):
        if rnd == 0:
            eng.draft_level(0, feat, tok)
            for l in range(1, d):
                eng.draft_level(l)
        tree = eng.rerank_build_tree()
        nz = eng.node_logits(feat)
        T = (nz + torch.randn(nz.shape, device=dev, generator=torch.Generator(device=dev).manual_seed(rnd))).contiguous()
        ver = eng.verify_greedy(tree["tokens"], tree["parents"], T)
        F = g(torch.from_numpy(rng.standard_normal((B, n, h)).astype(np.float32)).to(fdt))
        path = torch.empty(B, d + 1, h, dtype=fdt, device=dev)
        nfeat, ntok = eng.extend(F, ver["accept_len"], ver["accept_nodes"], ver["accept_tokens"], path_fhat=path)
        torch.cuda.synchronize()
        al, an, at = map(to_np, (ver["accept_len"], ver["accept_nodes"], ver["accept_tokens"]))
        for b in range(B):
            assert torch.equal(nfeat[b].cpu(), F[b, an[b, al[b]]].cpu())
            assert int(ntok[b]) == at[b, al[b]]
        for l in range(1, d):
            eng.draft_level(l)
        # a fresh handle drafts the whole tree from the same root
        fresh.draft_level(0, nfeat.contiguous(), ntok)
        for l in range(1, d):
            fresh.draft_level(l)
        t_loop = eng.rerank_build_tree()
        t_new = fresh.rerank_build_tree()
        torch.cuda.synchronize()
        for key in ("tokens", "parents", "positions", "mask", "logscore"):
            assert torch.equal(t_loop[key], t_new[key]), (rnd, key)
        # oracle: the path rows and the next level 0
        if rnd == 1:
            ref = oracle.draft_extend(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, F.cpu(), al, an, at, d, w.topk,
                                      w.is_bf16)
            got = path.float().cpu().numpy()
            tol = np.abs(ref["path_fhat"]) * (2.0 ** -7 if w.is_bf16 else 1e-5) + 1e-5
            assert np.all(np.abs(got - ref["path_fhat"]) <= tol)
        feat = nfeat.contiguous()
        tree = t_loop
    eng.status()
    eng.close()
    fresh.close()


def test_extend_level_zero_logits_and_ids_match_the_oracle(dev):
    w = synth.custom(128, 2000, 4, 3, 4, 12, dtype="bf16")
    inp, eng = make(dev, w)
    g = lambda t: t.to(dev).contiguous()
    B, n, d, h, V, k = w.batch, w.num_nodes, w.depth, w.hidden, w.vocab, w.topk
    rng = np.random.default_rng(5)
    F = torch.from_numpy(rng.standard_normal((B, n, h)).astype(np.float32)).to(torch.bfloat16)
    al = rng.integers(0, d + 1, size=B).astype(np.int32)
    an = -np.ones((B, d + 1), np.int32)
    at = -np.ones((B, d + 1), np.int32)
    for b in range(B):
        an[b, :al[b] + 1] = [0] + sorted(rng.choice(np.arange(1, n), size=al[b], replace=False).tolist())
        at[b, :al[b] + 1] = rng.integers(0, V, size=al[b] + 1)
    logits = torch.empty(B, V, dtype=torch.float32, device=dev)
    ti = lambda a: torch.from_numpy(a).to(dev)
    eng.extend(g(F), ti(al), ti(an), ti(at), logits_out=logits)
    v = eng.views()
    torch.cuda.synchronize()
    ref = oracle.draft_extend(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, F, al, an, at, d, k, True)
    z = to_np(logits)
    zr = np.stack([ref["path_z"][b, al[b]] for b in range(B)])
    assert np.max(np.abs(z - zr)) <= BF16_ABS
    ids = to_np(v["row_ids"])[:B]
    dev_z = float(np.max(np.abs(z - zr)))
    for b in range(B):
        srt = np.sort(zr[b])[::-1]
        margins = -np.diff(srt[:k + 1])
        if margins.min() > 2 * dev_z + 1e-6:
            assert ids[b].tolist() == ref["ids"][b].tolist()
    eng.close()
