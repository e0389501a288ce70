"""The draft decoder layer on the GPU (eagle_decoder_layer) against the oracle's orc_decoder_layer.

Both sides round at the same points (each projection's output, the attention output, both residual
sums, the normed activation, the MLP product); they differ in fp32 summation order, which can move a
bf16 rounding by one ulp.  So each output is checked (1) within the layer's bf16 tolerance of a
float64 torch restatement, the bound the oracle itself is pinned to, (2) within twice that bound of
the oracle, and (3) bit-identical to the oracle for most elements.  The tree's new values (one projection) are within one
bf16 ulp of the oracle's plus the fp32 summation-order slack of the projection; the new keys,
rotated after rounding, within the same carried through the rotation.

At the 7B draft layer's sizes the oracle runs on sampled nodes: a node's output depends on its
ancestors only (the tree mask), so the oracle takes the chain root..node of a sampled node as a
tree of its own and its last output is compared with the GPU's output for that node.
"""
import numpy as np
import pytest
import torch

import oracle
from decoder_ref import layer, random_tree, reference_layer, tolerance, tree_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    return torch.device("cuda", 0)


def gpu_layer(dev, w, d, masks, pos, new_kv=True):
    from eagle_speculative_decoding_draft_gb300.engine import DecoderLayer
    g = lambda t: t.to(dev).contiguous()
    lay = DecoderLayer(g(w["w_qkv"]), g(w["w_o"]), g(w["w_norm"]), g(w["w_gu"]), g(w["w_d"]), d["H"], d["Hk"])
    P = d["P"]
    res = lay(g(w["x"]), g(w["k_cache"]) if P else None, g(w["v_cache"]) if P else None,
              torch.as_tensor(pos, dtype=torch.int32).to(dev), torch.as_tensor(masks.view(np.int32)).to(dev),
              new_kv=new_kv)
    torch.cuda.synchronize()
    if new_kv:
        return [t.float().cpu().numpy() for t in res]
    return res.float().cpu().numpy()


def proj_abs(x, W):
    """sum_i |W[o][i]| |x[..., i]| in float64: the size of a projection's summands."""
    return (x.double().abs() @ W.double().abs().T).numpy()


def accum_slack(K, A):
    """fp32 accumulation of K summands whose absolute sum is A, in any order, ends within
    K * 2^-24 * A of the exact sum (2^-23 for an accumulator that truncates); the two sides
    together within K * 2^-22 * A."""
    return K * 2.0 ** -22 * A


def ulp_close(a, b, slack):
    """Values (one rounded projection): within one bf16 ulp of the larger magnitude (a rounding
    that the summation order moved) plus the summation slack; returns (ok, share equal)."""
    tol = 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + slack + 1e-30
    return bool(np.all(np.abs(a - b) <= tol)), float(np.mean(a == b))


def keys_close(a, b, slack):
    """Rotated keys: each input of a rotated pair (j, j + D/2) is within one ulp (at most 2^-7 times
    the pair's norm, which the rotation keeps) plus its summation slack; the rotation moves each
    output by at most the sum of both inputs' errors; then one ulp of the output's own rounding."""
    half = a.shape[-1] // 2
    r = np.sqrt(a[..., :half] ** 2 + a[..., half:] ** 2)
    r = np.concatenate([r, r], axis=-1)
    sl = slack[..., :half] + slack[..., half:]
    sl = np.concatenate([sl, sl], axis=-1)
    tol = 2.0 ** -7 * (2 * r + np.maximum(np.abs(a), np.abs(b))) + sl + 1e-30
    return bool(np.all(np.abs(a - b) <= tol)), float(np.mean(a == b))


def kv_slack(x, w, d):
    """Summation slack of the key and value projections of the rows of x, shaped [..., Hkv, D]."""
    H, Hk, D, h = d["H"], d["Hk"], d["D"], d["h"]
    shape = tuple(x.shape[:-1]) + (Hk, D)
    ak = proj_abs(x, w["w_qkv"][H * D:(H + Hk) * D]).reshape(shape)
    av = proj_abs(x, w["w_qkv"][(H + Hk) * D:]).reshape(shape)
    return accum_slack(h, ak), accum_slack(h, av)


def check_kv(kn, vn, k_orc, v_orc, slack_k, slack_v):
    ok, share = keys_close(kn, k_orc, slack_k)
    assert ok and share >= 0.95, ("k_new", ok, share)
    ok, share = ulp_close(vn, v_orc, slack_v)
    assert ok and share >= 0.95, ("v_new", ok, share)


def check_out(got, orc, ref, h1, absterms, exact_share=0.75):
    bound = tolerance(h1, ref, absterms)
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))
    assert np.all(np.abs(got - orc) <= 2 * bound), float(np.max(np.abs(got - orc) - 2 * bound))
    assert np.mean(got == orc) >= exact_share, float(np.mean(got == orc))


CASES = [
    # B, n, P, h, H, Hk, D, I, max_depth
    (2, 9, 37, 256, 4, 2, 64, 512, 4),      # GQA, several GEMM tiles, ragged key block
    (1, 1, 0, 128, 2, 2, 128, 256, 0),      # a lone root, no cache, MHA, D = 128
    (3, 40, 70, 192, 3, 1, 32, 320, 6),     # two mask words, MQA, ragged everywhere
    (4, 80, 5, 256, 4, 4, 64, 384, 6),      # 320 rows: two GEMM row chunks, deferred split-K sums
    (40, 4, 300, 128, 8, 8, 128, 256, 3),   # 16 query rows a CTA, D = 128, 5 key tiles each (no key split)
    (2, 8, 700, 128, 2, 2, 128, 256, 4),    # the same rows split over the keys: runs of 2 tiles
    (3, 3, 150, 128, 4, 2, 64, 256, 2),     # 6 query rows of 2-head groups, D = 64, key splits
    (2, 4, 90, 64, 2, 1, 32, 128, 3),       # exactly 8 query rows (MQA pairs), D = 32
    (2, 1, 130, 128, 8, 1, 64, 256, 0),     # a lone root under 8-head groups: 8 query rows of one node
    # more than 64 query rows per (request, kv head) with D = 64 or 128: the tcgen05 kernel
    (2, 40, 200, 256, 8, 2, 128, 512, 5),   # 160 rows (two 128-row tiles), ragged keys, key splits
    (3, 33, 1000, 256, 4, 1, 128, 512, 6),  # MQA, 132 rows, a tile of cached and tree keys, 8 splits
    (16, 30, 64, 128, 8, 2, 128, 256, 4),   # 120 rows, two key tiles, no key split
    (2, 50, 129, 128, 4, 2, 64, 256, 5),    # D = 64, 100 rows, three key tiles split
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_n%d_P%d_h%d_H%d_Hk%d_D%d" % c[:7])
def test_layer_matches_the_oracle(dev, case):
    B, n, P, h, H, Hk, D, I, md = case
    rng = np.random.default_rng(n * 7 + P)
    w, d = layer(B=B, n=n, P=P, h=h, H=H, Hk=Hk, D=D, I=I, seed=n + P, fan_in=True)
    trees = [random_tree(n, md, rng) for _ in range(B)]
    masks = np.stack([tree_mask(t[0]) for t in trees])
    pos = np.array([[P + dep for dep in t[1]] for t in trees], np.int32)
    out, kn, vn = gpu_layer(dev, w, d, masks, pos)
    orc = oracle.decoder_layer(w["x"], w["w_qkv"], w["w_o"], w["w_norm"], w["w_gu"], w["w_d"], w["k_cache"],
                               w["v_cache"], pos, masks, H, Hk, new_kv=True)
    for b in range(B):
        wb = {k: v[b:b + 1] if k in ("x", "k_cache", "v_cache") else v for k, v in w.items()}
        ref, h1, absterms = reference_layer(wb, dict(d, B=1), trees[b][0], pos[b:b + 1])
        check_out(out[b:b + 1], orc["out"][b:b + 1], ref, h1, absterms)
    check_kv(kn, vn, orc["k_new"], orc["v_new"], *kv_slack(w["x"], w, d))


def test_arbitrary_positions_and_a_full_mask_word(dev):
    """Positions that are not prefix + depth, and exactly 32 nodes (one full mask word)."""
    B, n, P = 2, 32, 11
    rng = np.random.default_rng(5)
    w, d = layer(B=B, n=n, P=P, h=128, H=2, Hk=1, D=64, I=256, seed=3, fan_in=True)
    trees = [random_tree(n, 5, rng) for _ in range(B)]
    masks = np.stack([tree_mask(t[0]) for t in trees])
    pos = rng.integers(0, 5000, size=(B, n)).astype(np.int32)
    out = gpu_layer(dev, w, d, masks, pos, new_kv=False)
    orc = oracle.decoder_layer(w["x"], w["w_qkv"], w["w_o"], w["w_norm"], w["w_gu"], w["w_d"], w["k_cache"],
                               w["v_cache"], pos, masks, 2, 1)["out"]
    for b in range(B):
        wb = {k: v[b:b + 1] if k in ("x", "k_cache", "v_cache") else v for k, v in w.items()}
        ref, h1, absterms = reference_layer(wb, dict(d, B=1), trees[b][0], pos[b:b + 1])
        check_out(out[b:b + 1], orc[b:b + 1], ref, h1, absterms)


def test_nodes_outside_the_ancestry_do_not_change_an_output(dev):
    """The mask decides visibility: changing a leaf's input changes no other node's output."""
    B, n, P = 1, 12, 20
    rng = np.random.default_rng(9)
    w, d = layer(B=B, n=n, P=P, h=128, H=4, Hk=2, D=32, I=256, seed=4, fan_in=True)
    parents, depths = random_tree(n, 4, rng)
    leaf = max(i for i in range(n) if i not in parents)
    masks = tree_mask(parents)[None]
    pos = np.array([[P + x for x in depths]], np.int32)
    base = gpu_layer(dev, w, d, masks, pos, new_kv=False)
    w2 = dict(w)
    x = w["x"].clone()
    x[:, leaf] = x[:, leaf] * -2 + 0.5
    w2["x"] = x
    got = gpu_layer(dev, w2, d, masks, pos, new_kv=False)
    others = [i for i in range(n) if i != leaf]
    assert np.array_equal(got[:, others], base[:, others])
    assert not np.array_equal(got[:, leaf], base[:, leaf])


def test_empty_batch_is_a_no_op(dev):
    from eagle_speculative_decoding_draft_gb300.engine import DecoderLayer
    w, d = layer(B=1, n=3, P=2, h=64, H=2, Hk=2, D=32, I=64, fan_in=True)
    g = lambda t: t.to(dev).contiguous()
    lay = DecoderLayer(g(w["w_qkv"]), g(w["w_o"]), g(w["w_norm"]), g(w["w_gu"]), g(w["w_d"]), 2, 2)
    x = torch.empty(0, 3, 64, dtype=torch.bfloat16, device=dev)
    out = lay(x, None, None, torch.empty(0, 3, dtype=torch.int32, device=dev),
              torch.empty(0, 3, 1, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert out.shape == (0, 3, 64)


def sampled_chains(dev, B, n, P, h, H, Hk, D, I, depth, seed, picks, exact_share):
    """The layer over B requests of an n-node tree each; for `picks` (request, node) pairs the
    oracle runs the chain root..node as a tree of its own and its last output is compared with
    the GPU's output for that node."""
    rng = np.random.default_rng(seed)
    w, d = layer(B=B, n=n, P=P, h=h, H=H, Hk=Hk, D=D, I=I, seed=seed % 97, fan_in=True)
    trees = [random_tree(n, depth, rng) for _ in range(B)]
    masks = np.stack([tree_mask(t[0]) for t in trees])
    pos = np.array([[P + dep for dep in t[1]] for t in trees], np.int32)
    out, kn, vn = gpu_layer(dev, w, d, masks, pos)
    for b, node in picks(trees, rng):
        parents = trees[b][0]
        chain = [node]
        while parents[chain[-1]] >= 0:
            chain.append(parents[chain[-1]])
        chain = chain[::-1]
        m = len(chain)
        wc = dict(w)
        wc["x"] = w["x"][b:b + 1, chain].contiguous()
        wc["k_cache"], wc["v_cache"] = w["k_cache"][b:b + 1], w["v_cache"][b:b + 1]
        cpar = [-1] + list(range(m - 1))
        cpos = pos[b:b + 1, chain]
        orc = oracle.decoder_layer(wc["x"], w["w_qkv"], w["w_o"], w["w_norm"], w["w_gu"], w["w_d"],
                                   wc["k_cache"], wc["v_cache"], cpos, tree_mask(cpar)[None], H, Hk,
                                   new_kv=True)
        ref, h1, absterms = reference_layer(wc, dict(d, B=1, n=m), cpar, cpos)
        check_out(out[b:b + 1, node:node + 1], orc["out"][:, -1:], ref[:, -1:], h1[:, -1:],
                  absterms[:, -1:], exact_share=exact_share)
        sk, sv = kv_slack(w["x"][b, node], w, d)
        check_kv(kn[b, node], vn[b, node], orc["k_new"][0, -1], orc["v_new"][0, -1], sk, sv)


def test_7b_draft_layer_on_sampled_nodes(dev):
    """Vicuna-7B draft layer sizes (h 4096, 32 heads of 128, MLP 11008), a 1024-token cache and a
    61-node tree of depth 6 per request; the oracle checks sampled nodes through their chains.
    At these sizes (sums over 4096 and 11008 terms) the summation order moves the bf16 rounding of
    a few percent of the MLP's gate and up values; the down projection gathers ~10^3 such one-ulp
    moves per output, about a third of an output ulp, so about a quarter of the outputs round the
    other way (72% equal measured)."""
    def picks(trees, rng):
        for b in range(len(trees)):
            depths = trees[b][1]
            yield b, max(range(len(depths)), key=lambda i: depths[i])
            yield b, int(rng.integers(1, len(depths)))
    sampled_chains(dev, B=2, n=61, P=1024, h=4096, H=32, Hk=32, D=128, I=11008, depth=6, seed=61,
                   picks=picks, exact_share=0.5)


def test_projections_over_several_row_chunks(dev):
    """366 node rows (6 requests x 61 nodes): every projection runs as one launch over two row
    chunks of 256 (the second ragged, 110 rows), grouped-query heads; nodes are sampled in both
    chunks, including the last row."""
    def picks(trees, rng):
        yield 0, 1
        yield 3, 60   # row 243, first chunk
        yield 4, 20   # row 264, second chunk
        yield 5, 60   # row 365, the last
        yield 5, int(rng.integers(1, 61))
    sampled_chains(dev, B=6, n=61, P=256, h=1024, H=16, Hk=4, D=64, I=2816, depth=6, seed=366,
                   picks=picks, exact_share=0.5)


def test_small_activations_where_the_norm_epsilon_counts(dev):
    """Inputs near 1e-3: the mean square of h1 is near the epsilon, which then moves the normed
    activation by a large factor."""
    B, n, P = 2, 7, 9
    rng = np.random.default_rng(11)
    w, d = layer(B=B, n=n, P=P, h=128, H=2, Hk=2, D=64, I=256, seed=6, fan_in=True)
    w["x"] = (w["x"].float() * 1e-3).to(torch.bfloat16)
    trees = [random_tree(n, 3, rng) for _ in range(B)]
    masks = np.stack([tree_mask(t[0]) for t in trees])
    pos = np.array([[P + dep for dep in t[1]] for t in trees], np.int32)
    out = gpu_layer(dev, w, d, masks, pos, new_kv=False)
    orc = oracle.decoder_layer(w["x"], w["w_qkv"], w["w_o"], w["w_norm"], w["w_gu"], w["w_d"], w["k_cache"],
                               w["v_cache"], pos, masks, 2, 2)["out"]
    for b in range(B):
        wb = {k: v[b:b + 1] if k in ("x", "k_cache", "v_cache") else v for k, v in w.items()}
        ref, h1, absterms = reference_layer(wb, dict(d, B=1), trees[b][0], pos[b:b + 1])
        check_out(out[b:b + 1], orc[b:b + 1], ref, h1, absterms)
