"""Pins of the oracle's draft-tree step (expand, rerank, tree build) against what the pages fix.

* a float64 restatement that computes every node's row by recursion along its token path
  (feature of a node = FC of its parent row's output and its own token) and applies the
  expand / rerank selection with full sorts; it shares none of the oracle's row/slot/candidate
  bookkeeping, so a feature routed to the wrong row, a wrong token, a dropped bias or a wrong
  score accumulation fails it;
* the two properties stated for EAGLE-2's expand + rerank (child value <= parent value, the
  kept top-m set is a connected tree, ties to the shallower node);
* the ancestor-only mask against a transitive closure computed by Warshall's algorithm, and
  positions equal to depth;
* topk = 1 degenerates to the greedy chain obtained by direct recursion.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from eagle_speculative_decoding_draft_gb300 import synth


def small_workload(h, V, B, d, k, m, dtype, bias=True, seed=0):
    w = synth.custom(h, V, B, d, k, m, dtype=dtype, bias=bias)
    return w, synth.make_inputs(w, seed=seed)


def run_oracle(w, inp, **kw):
    return oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok,
                             w.depth, w.topk, w.num_keep, w.is_bf16, **kw)


def f64(t):
    return t.double().numpy()


def bf16_round64(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


# ------------------------------------------------------------------------------------------
# float64 restatement by path recursion
# ------------------------------------------------------------------------------------------

def restated_tree(w, inp, b):
    Wfc, bfc, Wlm, E = f64(inp.w_fc), f64(inp.b_fc), f64(inp.w_lm), f64(inp.emb)
    k, d, m = w.topk, w.depth, w.num_keep
    margins = []

    def row(feat, tok):
        y = Wfc @ np.concatenate([feat, E[tok]]) + bfc
        fh = bf16_round64(y) if w.is_bf16 else y
        z = Wlm @ fh
        lse = logsumexp(z)
        order = np.lexsort((np.arange(z.shape[0]), -z))
        if z.shape[0] > k:
            margins.append(z[order[k - 1]] - z[order[k]])
        ids = order[:k]
        return fh, ids, z[ids] - lse

    root_fh, ids, logp = row(f64(inp.root_feat)[b], int(inp.root_tok[b]))
    level = [((int(t),), float(s), root_fh) for t, s in zip(ids, logp)]
    pool = list(level)
    frontier = level
    for l in range(2, d + 1):
        children = []
        for path, S, feat_in in frontier:
            fh, ids, logp = row(feat_in, path[-1])
            children += [(path + (int(t),), S + float(s), fh) for t, s in zip(ids, logp)]
        pool += children
        if l < d:
            srt = sorted(children, key=lambda c: -c[1])
            if len(srt) > k:
                margins.append(srt[k - 1][1] - srt[k][1])
            frontier = srt[:k]
    srt = sorted(pool, key=lambda c: -c[1])
    if w.num_keep < len(srt):
        margins.append(srt[m - 1][1] - srt[m][1])
    kept = {c[0]: c[1] for c in srt[:m]}
    return kept, min(margins) if margins else np.inf


def oracle_paths(out, b):
    tok, par, S = out["tree_tok"][b], out["tree_parent"][b], out["tree_S"][b]
    paths = {}
    for i in range(1, tok.shape[0]):
        p, a = [], i
        while a != 0:
            p.append(int(tok[a]))
            a = par[a]
        paths[tuple(reversed(p))] = float(S[i])
    return paths


CASES = [
    dict(h=16, V=50, B=3, d=3, k=3, m=10, dtype="f32"),
    dict(h=16, V=50, B=3, d=3, k=3, m=10, dtype="bf16"),
    dict(h=24, V=80, B=2, d=4, k=2, m=14, dtype="bf16"),   # keeps the whole pool
    dict(h=8, V=30, B=2, d=5, k=4, m=25, dtype="f32"),
    dict(h=32, V=120, B=2, d=2, k=5, m=7, dtype="bf16"),
    dict(h=16, V=40, B=2, d=4, k=1, m=3, dtype="bf16"),    # chain, truncated
    dict(h=16, V=40, B=2, d=1, k=4, m=2, dtype="f32"),     # one level
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "h{h}V{V}B{B}d{d}k{k}m{m}{dtype}".format(**c))
def test_tree_equals_float64_path_recursion(case):
    w, inp = small_workload(case["h"], case["V"], case["B"], case["d"], case["k"], case["m"],
                            case["dtype"], seed=100 + case["h"] + case["d"])
    out = run_oracle(w, inp)
    for b in range(w.batch):
        kept, margin = restated_tree(w, inp, b)
        assert margin > 1e-4, "seed gives a near-tie; the comparison would not be decisive"
        got = oracle_paths(out, b)
        assert set(got) == set(kept)
        for p, s in kept.items():
            assert abs(got[p] - s) < 1e-4 * max(1.0, abs(s))


# ------------------------------------------------------------------------------------------
# structural properties of every tree
# ------------------------------------------------------------------------------------------

def warshall_closure(parent):
    n = parent.shape[0]
    A = np.eye(n, dtype=bool)
    for i in range(1, n):
        A[i, parent[i]] = True
    for kk in range(n):
        A = A | (A[:, [kk]] & A[[kk], :])
    return A


def unpack_mask(words, n):
    bits = np.zeros((words.shape[0], n), dtype=bool)
    for j in range(n):
        bits[:, j] = (words[:, j // 32] >> np.uint32(j % 32)) & np.uint32(1)
    return bits


PROP_CASES = [
    dict(h=64, V=3000, B=3, d=5, k=4, m=30, dtype="bf16"),
    dict(h=32, V=2000, B=2, d=6, k=10, m=60, dtype="bf16"),
    dict(h=48, V=700, B=2, d=5, k=8, m=64, dtype="f32"),
    dict(h=16, V=100, B=4, d=3, k=2, m=6, dtype="f32"),
    dict(h=16, V=300, B=1, d=16, k=16, m=600, dtype="bf16"),  # 3856 candidates, near the 4096 cap
    dict(h=16, V=100, B=1, d=32, k=11, m=300, dtype="f32"),   # the deepest tree the API takes
]


@pytest.mark.parametrize("case", PROP_CASES, ids=lambda c: "d{d}k{k}m{m}{dtype}".format(**c))
def test_tree_properties(case):
    w, inp = small_workload(case["h"], case["V"], case["B"], case["d"], case["k"], case["m"],
                            case["dtype"], seed=7)
    pos_base = np.arange(w.batch, dtype=np.int32) * 100 + 5
    out = run_oracle(w, inp, pos_base=pos_base)
    k, d, m, n = w.topk, w.depth, w.num_keep, w.num_keep + 1
    nc = w.num_candidates
    for b in range(w.batch):
        par, tok, pos, S = (out["tree_parent"][b], out["tree_tok"][b], out["tree_pos"][b],
                            out["tree_S"][b])
        cand = out["tree_cand"][b]
        assert par[0] == -1 and tok[0] == int(inp.root_tok[b]) and S[0] == 0.0
        depth = np.zeros(n, int)
        for i in range(1, n):
            assert 0 <= par[i] < i  # topological, level-major order
            depth[i] = depth[par[i]] + 1
            assert S[i] <= S[par[i]]  # value(child) <= value(parent)
        assert np.all(np.diff(depth) >= 0)
        assert np.array_equal(pos, depth + pos_base[b])
        assert depth.max() <= d
        # ancestor-only mask == transitive closure of the parent relation
        assert np.array_equal(unpack_mask(out["tree_mask"][b], n), warshall_closure(par))
        # siblings carry distinct tokens
        for i in range(n):
            kids = tok[par == i]
            assert len(set(kids.tolist())) == len(kids)
        # the kept set is exactly the top-m of the pool by (S desc, candidate asc)
        cS = out["cand_S"][b]
        order = sorted(range(nc), key=lambda c: (-cS[c], c))
        assert sorted(cand[1:].tolist()) == sorted(order[:m])
        assert np.array_equal(cand[1:], np.sort(cand[1:]))
        # pool scores: S(child) = fl32(S(parent) + logp), and the closed form sum of logp
        cpar, crow = out["cand_parent"][b], out["cand_row"][b]
        for c in range(nc):
            lvl = 0 if c < k else 1 + (c - k) // (k * k)
            j = c % k if c < k else (c - k) % k
            logp = out["row_logp"][lvl, crow[c], j]
            assert out["row_ids"][lvl, crow[c], j] == out["cand_tok"][b, c]
            parent_S = np.float32(0.0) if cpar[c] < 0 else cS[cpar[c]]
            assert cS[c] == np.float32(parent_S + logp)
        # frontier of each level = top-k of the previous level's k^2 by (S desc, cand asc)
        for lvl in range(2, d):
            base = k + (lvl - 2) * k * k
            ids = list(range(base, base + k * k))
            ref = sorted(ids, key=lambda c: (-cS[c], c))[:k]
            assert out["front_cand"][lvl, b].tolist() == ref


def test_keep_everything_and_keep_nothing():
    w, inp = small_workload(16, 60, 2, 3, 3, 21, "bf16", seed=4)
    out = run_oracle(w, inp)
    assert np.array_equal(out["tree_cand"][:, 1:], np.tile(np.arange(21), (2, 1)))
    w0 = w.replace(num_keep=0)
    out0 = run_oracle(w0, inp)
    assert out0["tree_tok"].shape == (2, 1) and np.all(out0["tree_parent"] == -1)


# ------------------------------------------------------------------------------------------
# topk = 1: the tree is the greedy chain obtained by direct recursion
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,m", [(4, 4), (5, 3), (3, 7)])
def test_topk1_is_the_greedy_chain(dtype, d, m):
    m = min(m, d)
    w, inp = small_workload(24, 90, 2, d, 1, m, dtype, seed=31)
    out = run_oracle(w, inp)
    for b in range(w.batch):
        feat = inp.root_feat[b].float().numpy()
        tok = int(inp.root_tok[b])
        chain = []
        for _ in range(d):
            fh = oracle.fc_row(inp.w_fc, inp.b_fc, feat, inp.emb, tok, w.is_bf16)
            z = oracle.lm_head_row(inp.w_lm, fh, w.is_bf16)
            tok = int(np.lexsort((np.arange(z.shape[0]), -z))[0])
            chain.append(tok)
            feat = fh
        assert out["tree_tok"][b, 1:].tolist() == chain[:m]
        assert out["tree_parent"][b].tolist() == list(range(-1, m))


# ------------------------------------------------------------------------------------------
# node logits (synthetic target rows): each node's own row, by recursion along its path
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_node_logits_follow_each_nodes_path(dtype):
    w, inp = small_workload(16, 70, 2, 4, 3, 12, dtype, seed=17)
    out = run_oracle(w, inp, row_logits=True, node_logits=True)
    for b in range(w.batch):
        tok, par = out["tree_tok"][b], out["tree_parent"][b]
        feat_in = {0: inp.root_feat[b].float().numpy()}
        for i in range(w.num_nodes):  # parents come first (level-major order)
            if i > 0:
                # the input feature of node i is the output of its parent's own row
                feat_in[i] = oracle.fc_row(inp.w_fc, inp.b_fc, feat_in[par[i]], inp.emb,
                                           int(tok[par[i]]), w.is_bf16)
            fh = oracle.fc_row(inp.w_fc, inp.b_fc, feat_in[i], inp.emb, int(tok[i]), w.is_bf16)
            z = oracle.lm_head_row(inp.w_lm, fh, w.is_bf16)
            assert np.array_equal(out["node_z"][b, i], z)
        # the root's row is level 0's row b
        assert np.array_equal(out["node_z"][b, 0], out["row_z"][0, b])
