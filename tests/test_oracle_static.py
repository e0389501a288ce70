"""Pins of the oracle's EAGLE-1 static tree (orc_draft_static).

"EAGLE 推测解码为什么比 Medusa 快？" (chapter 04 notes) §10.1 and §12 item 7: EAGLE-1 drafts a tree
of fixed shape (set by position only); node j is (parent, rank): the rank-th most probable draft
token at its parent.  Pinned by the dynamic tree's special cases (a rank-0 chain is the dynamic
tree with topk = 1; a star of the top k is depth 1 with m = k) and by a full binary tree built
here from the row functions.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_draft_gb300 import synth


def test_rank_zero_chain_is_the_topk_one_tree():
    w = synth.custom(64, 300, 3, 5, 1, 5, dtype="bf16")
    inp = synth.make_inputs(w, seed=2)
    spec = [[j, 0] for j in range(w.depth)]
    s = oracle.draft_static(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok, spec, True)
    t = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok, w.depth, 1,
                          w.depth, True)
    for key in ("tree_tok", "tree_parent", "tree_pos", "tree_mask", "tree_S"):
        assert np.array_equal(s[key], t[key]), key


def test_top_k_star_is_the_depth_one_tree():
    w = synth.custom(64, 300, 4, 1, 5, 5, dtype="bf16")
    inp = synth.make_inputs(w, seed=4)
    spec = [[0, r] for r in range(w.topk)]
    pos = np.arange(w.batch, dtype=np.int32) * 7
    s = oracle.draft_static(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok, spec, True,
                            pos_base=pos)
    t = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok, 1, w.topk,
                          w.topk, True, pos_base=pos)
    for key in ("tree_tok", "tree_parent", "tree_pos", "tree_mask", "tree_S"):
        assert np.array_equal(s[key], t[key]), key


def test_full_binary_tree_by_composition():
    w = synth.WORKLOADS[1]  # fp32, h 256, V 1024
    inp = synth.make_inputs(w, seed=6)
    # root -> 1, 2 (ranks 0, 1); 1 -> 3, 4; 2 -> 5, 6
    spec = [[0, 0], [0, 1], [1, 0], [1, 1], [2, 0], [2, 1]]
    s = oracle.draft_static(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok, spec, False,
                            node_fhat=True)
    W_fc, W_lm, E = (x.numpy() for x in (inp.w_fc, inp.w_lm, inp.emb))
    bias = inp.b_fc.numpy() if inp.b_fc is not None else None

    def row(feat, tok):
        fh = oracle.fc_row(W_fc, bias, feat.astype(np.float32), E, int(tok), False)
        z = oracle.lm_head_row(W_lm, fh, False)
        ids, logp, _ = oracle.log_softmax_topk(z, 2)
        return fh, ids, logp

    for b in range(w.batch):
        f0 = inp.root_feat[b].numpy()
        fh0, ids0, lp0 = row(f0, inp.root_tok[b])
        toks = {1: ids0[0], 2: ids0[1]}
        S = {1: lp0[0], 2: lp0[1]}
        fhs = {0: fh0}
        for parent, (c0, c1) in ((1, (3, 4)), (2, (5, 6))):
            fh, ids, lp = row(fh0, toks[parent])
            fhs[parent] = fh
            toks[c0], toks[c1] = ids[0], ids[1]
            S[c0] = np.float32(S[parent]) + np.float32(lp[0])
            S[c1] = np.float32(S[parent]) + np.float32(lp[1])
        assert s["tree_tok"][b].tolist() == [int(inp.root_tok[b])] + [int(toks[j]) for j in range(1, 7)]
        assert s["tree_parent"][b].tolist() == [-1, 0, 0, 1, 1, 2, 2]
        assert s["tree_pos"][b].tolist() == [0, 1, 1, 2, 2, 2, 2]
        assert s["tree_mask"][b].ravel().tolist() == [0b1, 0b11, 0b101, 0b1011, 0b10011, 0b100101, 0b1000101]
        assert np.array_equal(s["tree_S"][b][1:], np.array([S[j] for j in range(1, 7)], np.float32))
        for j in (0, 1, 2):
            assert np.array_equal(s["node_fhat"][b, j], fhs[j])
        assert not s["node_fhat"][b, 3:].any()


@pytest.mark.parametrize("spec", [[[1, 0]], [[0, 0], [0, 0]], [[0, 0], [1, 0], [0, 1]], [[0, 16]]])
def test_rejects_malformed_shapes(spec):
    w = synth.WORKLOADS[1]
    inp = synth.make_inputs(w)
    with pytest.raises(RuntimeError):
        oracle.draft_static(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok, spec, False)
