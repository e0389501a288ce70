"""Pins of the oracle's draft extend (orc_draft_extend).

zdszero, "在 SGLang 里": after the verify the draft runs again over the verified positions with
the target's true hidden states and the accepted tokens; the last verified position starts the
next round and its top-k is the next round's first level.  The rows are checked against a
float64 restatement built here (not the oracle's C), the next root against the path, and the
last row against the oracle's own level 0 for that root.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_draft_gb300 import synth

U32 = 2.0 ** -24


def gamma(n):
    return n * U32 / (1 - n * U32)


def widen(t):
    return t.float().numpy().astype(np.float64) if hasattr(t, "float") else np.asarray(t, np.float64)


def random_paths(rng, B, n, d, V):
    al = rng.integers(0, d + 1, size=B).astype(np.int32)
    an = -np.ones((B, d + 1), np.int32)
    at = -np.ones((B, d + 1), np.int32)
    for b in range(B):
        nodes = [0] + sorted(rng.choice(np.arange(1, n), size=al[b], replace=False).tolist())
        an[b, :al[b] + 1] = nodes
        at[b, :al[b] + 1] = rng.integers(0, V, size=al[b] + 1)
    return al, an, at


@pytest.mark.parametrize("wl", [1, "bf16"])
def test_rows_follow_the_accepted_path(wl):
    if wl == 1:
        w = synth.WORKLOADS[1]
    else:
        w = synth.custom(64, 300, 3, 4, 3, 9, dtype="bf16")
    inp = synth.make_inputs(w, seed=3)
    rng = np.random.default_rng(7)
    B, n, d, h, V = w.batch, w.num_nodes, w.depth, w.hidden, w.vocab
    fdt = torch.bfloat16 if w.is_bf16 else torch.float32
    F = torch.from_numpy(rng.standard_normal((B, n, h)).astype(np.float32)).to(fdt)
    al, an, at = random_paths(rng, B, n, d, V)
    r = oracle.draft_extend(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, F, al, an, at, d, w.topk, w.is_bf16)
    Wfc, Wlm, E = widen(inp.w_fc), widen(inp.w_lm), widen(inp.emb)
    bias = widen(inp.b_fc) if inp.b_fc is not None else np.zeros(h)
    Fw = widen(F)
    for b in range(B):
        L = al[b]
        assert np.array_equal(r["next_feat"][b], Fw[b, an[b, L]].astype(np.float32))
        assert r["next_tok"][b] == at[b, L]
        for i in range(d + 1):
            j = min(i, L)
            x = np.concatenate([Fw[b, an[b, j]], E[at[b, j]]])
            fh = Wfc @ x + bias
            bound = gamma(2 * h + 1) * (np.abs(Wfc) @ np.abs(x) + np.abs(bias))
            if w.is_bf16:
                bound = bound + 2.0 ** -8 * (np.abs(fh) + bound)
            assert np.all(np.abs(r["path_fhat"][b, i] - fh) <= bound + 1e-30)
            # the LM head on the oracle's own f^ (exact inputs), within the fp32 dot bound
            fo = r["path_fhat"][b, i].astype(np.float64)
            z = Wlm @ fo
            zb = gamma(h) * (np.abs(Wlm) @ np.abs(fo))
            assert np.all(np.abs(r["path_z"][b, i] - z) <= zb + 1e-30)
            if i > L:
                assert np.array_equal(r["path_fhat"][b, i], r["path_fhat"][b, L])


def test_last_row_is_the_next_rounds_level_zero():
    w = synth.custom(64, 300, 4, 4, 3, 9, dtype="bf16")
    inp = synth.make_inputs(w, seed=5)
    rng = np.random.default_rng(11)
    B, n, d, h, V = w.batch, w.num_nodes, w.depth, w.hidden, w.vocab
    F = torch.from_numpy(rng.standard_normal((B, n, h)).astype(np.float32)).to(torch.bfloat16)
    al, an, at = random_paths(rng, B, n, d, V)
    r = oracle.draft_extend(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, F, al, an, at, d, w.topk, True)
    root_feat = torch.stack([F[b, an[b, al[b]]] for b in range(B)])
    root_tok = np.array([at[b, al[b]] for b in range(B)], np.int32)
    t = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, root_feat, root_tok, d, w.topk,
                          w.num_keep, True)
    for b in range(B):
        assert np.array_equal(r["path_fhat"][b, al[b]], t["row_fhat"][0][b])
        assert r["ids"][b].tolist() == t["row_ids"][0][b].tolist()
        assert np.array_equal(r["logp"][b], t["row_logp"][0][b])
        assert r["lse"][b] == t["row_lse"][0][b]


def test_rejects_broken_paths():
    w = synth.WORKLOADS[1]
    inp = synth.make_inputs(w)
    F = torch.zeros(1, w.num_nodes, w.hidden)
    d = w.depth
    with pytest.raises(RuntimeError):  # accept_len beyond the depth
        oracle.draft_extend(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, F, [d + 1], [[0] * (d + 1)],
                            [[1] * (d + 1)], d, w.topk, False)
    with pytest.raises(RuntimeError):  # a node outside the tree
        oracle.draft_extend(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, F, [1], [[0, w.num_nodes] + [-1] * (d - 1)],
                            [[1, 2] + [-1] * (d - 1)], d, w.topk, False)
