"""Component parity on the GPU, through the C ABI, against the oracle on identical inputs.

* streamed-weight GEMM (tcgen05): every output within the fp32 dot-product error bound of the
  oracle's fp32 dot product (both sides are within gamma_K * sum|w x| of the exact value), on
  ragged shapes (M, K not tile multiples, 1..256 rows) and bit-identical across launches;
* row log-softmax/top-k: ids bit-exact (same fp32 inputs, same tie rule), lse and logp within
  the fp32 summation bound, fp32 and bf16 inputs, strided rows;
* expand, rerank/build and the verify walk: bit-exact on the oracle's own intermediate arrays.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_draft_gb300 import synth
from parity import to_np

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from eagle_speculative_decoding_draft_gb300 import build, _lib
    build.build()
    _lib.load()
    return torch.device("cuda:0")


def gamma(n):
    return n * U32 / (1 - n * U32)


def bf16_tensor(rng, shape, std):
    return torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16)


# Ragged M and K, 1..256 rows (padded to the MMA's N in steps of 16), M below one 128-row tile.
# Above 16 rows every way of summing split tiles: the owner's fix-up with bulk stores when every
# worker covers a whole tile ((20000, 512), (20000, 520) with a ragged last k-block: 157 tiles,
# one CTA each) and the second launch otherwise ((4096, 8192) and (777, 1000): few tiles, long K;
# (70, 4104): one tile, ragged K).  With an even tile count the CTAs run as pairs (.cta_group::2,
# M = 256): (32000, 4096) at 17, 64 and 256 rows (the LM head: the owner's fix-up), (4096, 8192)
# at 256 rows and (2000, 2048, 128) (the FC's shape class: the second launch), (12000, 2048, 24),
# (130, 72, 255) (one pair of tiles split over two pairs with 255 rows, the largest ragged N) and
# (20480, 520, 40) (160 tiles, ragged last k-block).  More than 256 rows run as row chunks of 256
# in one launch: (1000, 520, 300) (CTA pairs, a 44-row last chunk), (777, 1000, 520) (odd tile
# count: single CTAs, an 8-row last chunk), (4096, 2048, 600) and (2048, 1024, 1100) (3 and 5
# chunks on CTA pairs).
LINEAR_CASES = [(128, 64, 1), (200, 200, 17), (1000, 512, 256), (300, 64, 33), (128, 128, 16),
                (4096, 8192, 10), (32000, 4096, 10), (777, 1000, 100), (130, 72, 255),
                (4096, 8192, 256), (300, 64, 64), (513, 1000, 49), (70, 4104, 80), (2000, 2048, 128),
                (20000, 512, 40), (20000, 520, 200), (12000, 2048, 24), (32000, 4096, 256),
                (32000, 4096, 17), (32000, 4096, 64), (20480, 520, 40),
                (1000, 520, 300), (777, 1000, 520), (4096, 2048, 600), (2048, 1024, 1100)]


@pytest.mark.parametrize("M,K,rows", LINEAR_CASES)
@pytest.mark.parametrize("out_bf16", [False, True])
def test_linear_within_fp32_bound_of_oracle(dev, M, K, rows, out_bf16):
    from eagle_speculative_decoding_draft_gb300.engine import linear_bf16
    rng = np.random.default_rng(M * 7 + K + rows)
    W = bf16_tensor(rng, (M, K), 1 / np.sqrt(K))
    X = bf16_tensor(rng, (rows, K), 1.0)
    bias = bf16_tensor(rng, (M,), 0.1)
    y = linear_bf16(W.to(dev), X.to(dev), bias.to(dev), out_bf16=out_bf16)
    y2 = linear_bf16(W.to(dev), X.to(dev), bias.to(dev), out_bf16=out_bf16)
    torch.cuda.synchronize()
    got = to_np(y.float()).astype(np.float64)
    assert np.array_equal(to_np(y.float()), to_np(y2.float())), "not deterministic"
    Wf = W.float().numpy().astype(np.float64)
    Xf = X.float().numpy()
    bf = bias.float().numpy().astype(np.float64)
    absdot = np.abs(Xf.astype(np.float64)) @ np.abs(Wf).T
    for r in range(rows):
        ref = oracle.lm_head_row(W, Xf[r], True).astype(np.float64) + bf
        bound = 2 * gamma(K + 1) * (absdot[r] + np.abs(bf)) + 1e-30
        if out_bf16:
            bound = bound + 2.0 ** -8 * (np.abs(ref) + bound)
        bad = np.abs(got[r] - ref) > bound
        assert not bad.any(), (r, np.argwhere(bad)[:3].ravel(), got[r][bad][:3], ref[bad][:3])


@pytest.mark.parametrize("M,K", [(4096, 8192), (32000, 4096), (300, 640)])
def test_linear_split_sums_do_not_depend_on_the_row_count(dev, M, K):
    """A row's result depends on the split of the k-blocks only, which is the same for every
    launch of 1-16 rows (stream-K, the last CTA of a split tile sums the partials) and for every
    launch of 17-256 rows (stream-K on single CTAs or CTA pairs, with the sum by the tile's
    owner or a second launch, both adding the same partials in the same CTA order)."""
    from eagle_speculative_decoding_draft_gb300.engine import linear_bf16
    rng = np.random.default_rng(M + K)
    W = bf16_tensor(rng, (M, K), 1 / np.sqrt(K)).to(dev)
    X = bf16_tensor(rng, (256, K), 1.0).to(dev)
    bias = bf16_tensor(rng, (M,), 0.1).to(dev)
    for out_bf16 in (False, True):
        one = linear_bf16(W, X[:1].contiguous(), bias, out_bf16=out_bf16)
        few = linear_bf16(W, X[:16].contiguous(), bias, out_bf16=out_bf16)
        more = linear_bf16(W, X[:17].contiguous(), bias, out_bf16=out_bf16)
        wide = linear_bf16(W, X[:64].contiguous(), bias, out_bf16=out_bf16)
        widest = linear_bf16(W, X, bias, out_bf16=out_bf16)
        torch.cuda.synchronize()
        assert torch.equal(one, few[:1])
        assert torch.equal(more, wide[:17])
        assert torch.equal(wide, widest[:64])


# At least as many rows as SMs, rows of 2^16 elements or more (and 16-byte aligned rows) take the
# streaming kernel: (200, 128256, 8), (160, 65536, 16) in bf16, (160, 70000, 1) with the
# logsumexp; their strided variants (row stride not a multiple of 16 bytes) the cluster one, as do
# (256, 32000, 4) (shorter rows).  The arg-max without the logsumexp streams from 32 KB rows on
# (test_verify_*).
TOPK_CASES = [(10, 32000, 10, "f32"), (3, 1000, 16, "f32"), (4, 128256, 8, "f32"),
              (5, 77, 4, "f32"), (2, 33, 1, "bf16"), (4, 5000, 2, "bf16"), (6, 1024, 2, "f32"),
              (300, 2048, 4, "f32"), (1, 16, 16, "f32"), (256, 32000, 4, "f32"), (200, 128256, 8, "f32"),
              (160, 65536, 16, "bf16"), (160, 70000, 1, "f32")]


@pytest.mark.parametrize("rows,V,k,dt", TOPK_CASES)
@pytest.mark.parametrize("strided", [False, True])
def test_row_topk_matches_oracle(dev, rows, V, k, dt, strided):
    from eagle_speculative_decoding_draft_gb300.engine import row_topk
    rng = np.random.default_rng(rows * 31 + V + k)
    z = (rng.standard_normal((rows, V)) * 2.1).astype(np.float32)
    z[::2] = np.round(z[::2] * 8) / 8  # exact ties on every other row
    zt = torch.from_numpy(z)
    if dt == "bf16":
        zt = zt.to(torch.bfloat16)
        z = zt.float().numpy()
    if strided:
        big = torch.zeros(rows, V + 3, dtype=zt.dtype)
        big[:, :V] = zt
        zd = big.to(dev)[:, :V]
    else:
        zd = zt.to(dev)
    ids, logp, lse = row_topk(zd, k, with_lse=True)
    am, raw, _ = row_topk(zd, 1, with_lse=False)
    torch.cuda.synchronize()
    ids, logp, lse, am, raw = map(to_np, (ids, logp, lse, am, raw))
    for r in range(rows):
        rid, rlogp, rlse = oracle.log_softmax_topk(z[r], k)
        assert ids[r].tolist() == rid.tolist()
        bound = gamma(V) * 2 + 8 * U32 * (1 + abs(rlse)) + 1e-6
        assert abs(lse[r] - rlse) <= bound
        assert np.all(np.abs(logp[r] - rlogp) <= bound + 8 * U32 * np.abs(rlogp))
        assert am[r, 0] == rid[0] and raw[r, 0] == z[r, rid[0]]


@pytest.mark.parametrize("V,k,dt", [(32000, 10, "f32"), (1000, 16, "f32"), (128256, 16, "f32"),
                                    (32000, 1, "bf16"), (4099, 7, "bf16"), (65536, 8, "bf16")])
def test_row_topk_massive_ties(dev, V, k, dt):
    """Thousands of entries tie at the top: the candidate lists overflow and every slice falls
    back to exact passes; ties go to the lower column.  With 160 rows of 2^16 elements or more
    the streaming kernel takes them: its warps' buffers fill with ties and settle them by column
    at each compaction."""
    from eagle_speculative_decoding_draft_gb300.engine import row_topk
    rng = np.random.default_rng(V + k)
    nrows = 160 if V >= 65536 and V % 8 == 0 else 4
    z = rng.integers(0, 3, size=(nrows, V)).astype(np.float32)
    z[1] = 0.0  # one constant row
    z[2, ::5] = 3.0
    zt = torch.from_numpy(z)
    if dt == "bf16":
        zt = zt.to(torch.bfloat16)
    ids, logp, lse = row_topk(zt.to(dev), k, with_lse=True)
    torch.cuda.synchronize()
    ids, logp, lse = map(to_np, (ids, logp, lse))
    for r in range(z.shape[0]):
        rid, rlogp, rlse = oracle.log_softmax_topk(z[r], k)
        assert ids[r].tolist() == rid.tolist()
        bound = gamma(V) * 2 + 8 * U32 * (1 + abs(rlse)) + 1e-6
        assert abs(lse[r] - rlse) <= bound
        assert np.all(np.abs(logp[r] - rlogp) <= bound + 8 * U32 * np.abs(rlogp))


def small_tree(dtype="bf16", B=3, d=4, k=3, m=12, h=32, V=300, seed=5):
    w = synth.custom(h, V, B, d, k, m, dtype=dtype)
    inp = synth.make_inputs(w, seed=seed)
    ref = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok,
                            d, k, m, w.is_bf16)
    return w, inp, ref


@pytest.mark.parametrize("B,d,k,m", [(3, 4, 3, 12), (2, 6, 10, 60), (5, 5, 4, 7), (4, 3, 1, 3),
                                     (2, 5, 16, 100), (1, 1, 4, 4),
                                     # the largest pools: 3856 candidates kept whole (3857 nodes,
                                     # 121 mask words), the deepest tree, a 32-level chain
                                     (2, 16, 16, 3856), (2, 32, 11, 3762), (2, 32, 11, 500), (1, 32, 1, 32)])
def test_expand_and_build_are_bit_exact_on_oracle_inputs(dev, B, d, k, m):
    from eagle_speculative_decoding_draft_gb300.engine import build_tree, expand
    w, inp, ref = small_tree(B=B, d=d, k=k, m=m, V=max(300, k + 1), seed=B + d + k)
    nc = w.num_candidates
    i32 = dict(dtype=torch.int32, device=dev)
    pool = {"tok": torch.full((B, nc), -7, **i32), "S": torch.zeros(B, nc, device=dev),
            "parent": torch.full((B, nc), -7, **i32), "row": torch.full((B, nc), -7, **i32)}
    R = B * k
    front_c = [torch.zeros(B, k, **i32) for _ in range(2)]
    front_s = [torch.zeros(B, k, device=dev) for _ in range(2)]
    for l in range(d):
        rows = B if l == 0 else R
        row_ids = torch.from_numpy(ref["row_ids"][l, :rows].copy()).to(dev)
        row_logp = torch.from_numpy(ref["row_logp"][l, :rows].copy()).to(dev)
        fin = None if l == 0 else (front_c[(l + 1) % 2], front_s[(l + 1) % 2])
        fout = (front_c[l % 2], front_s[l % 2]) if l < d - 1 else None
        expand(l, k, d, row_ids, row_logp, None if fin is None else fin[0],
               None if fin is None else fin[1], pool, fout)
        if l + 1 < d:
            torch.cuda.synchronize()
            assert to_np(front_c[l % 2]).tolist() == ref["front_cand"][l + 1].tolist()
    torch.cuda.synchronize()
    assert np.array_equal(to_np(pool["tok"]), ref["cand_tok"])
    assert np.array_equal(to_np(pool["S"]), ref["cand_S"])
    assert np.array_equal(to_np(pool["parent"]), ref["cand_parent"])
    assert np.array_equal(to_np(pool["row"]), ref["cand_row"])
    pos_base = torch.arange(B, dtype=torch.int32, device=dev) * 10 + 3
    status = torch.zeros(1, **i32)
    tree = build_tree(k, d, m, pool["tok"], pool["S"], pool["parent"], inp.root_tok.to(dev),
                      pos_base, status)
    torch.cuda.synchronize()
    ref_pb = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok,
                               d, k, m, w.is_bf16, pos_base=to_np(pos_base))
    assert np.array_equal(to_np(tree["tokens"]), ref_pb["tree_tok"])
    assert np.array_equal(to_np(tree["parents"]), ref_pb["tree_parent"])
    assert np.array_equal(to_np(tree["positions"]), ref_pb["tree_pos"])
    assert np.array_equal(to_np(tree["mask"]).astype(np.uint32), ref_pb["tree_mask"])
    assert np.array_equal(to_np(tree["logscore"]), ref_pb["tree_S"])
    assert int(status.item()) == 0


def test_verify_walk_and_greedy_are_bit_exact(dev):
    from eagle_speculative_decoding_draft_gb300.engine import row_topk, verify_walk
    rng = np.random.default_rng(99)
    B, n, V, d = 64, 10, 6, 9
    tok = np.zeros((B, n), np.int32)
    par = np.zeros((B, n), np.int32)
    for b in range(B):
        par[b, 0] = -1
        used = {}
        for i in range(1, n):
            p = int(rng.integers(0, i))
            par[b, i] = p
            t = int(rng.choice([v for v in range(V) if v not in used.setdefault(p, set())]))
            used[p].add(t)
            tok[b, i] = t
    T = rng.standard_normal((B, n, V)).astype(np.float32)
    for b in range(B):
        for i in range(n):
            kids = np.nonzero(par[b] == i)[0]
            if kids.size and rng.random() < 0.75:
                T[b, i, tok[b, rng.choice(kids)]] = 9.0
    ref = oracle.verify_greedy(tok, par, T, d)
    tt, pp = torch.from_numpy(tok).to(dev), torch.from_numpy(par).to(dev)
    g, _, _ = row_topk(torch.from_numpy(T).to(dev).view(B * n, V), 1, with_lse=False)
    out = verify_walk(tt, pp, g.view(B, n), d)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(g).reshape(B, n), ref["g"])
    assert np.array_equal(to_np(out["accept_len"]), ref["accept_len"])
    assert np.array_equal(to_np(out["accept_nodes"]), ref["accept_nodes"])
    assert np.array_equal(to_np(out["accept_tokens"]), ref["accept_tok"])
    assert ref["accept_len"].max() >= 3  # the planted agreements make long paths


@pytest.mark.parametrize("V", [6, 32000])
def test_verify_greedy_with_bf16_target_logits_is_bit_exact(dev, V):
    """eagle_verify_greedy on bf16 target logits (the dtype a bf16 target model emits): the
    arg-max over bf16 values, ties to the lowest id (rounding to bf16 makes ties common), against
    the oracle's walk over the same values widened to fp32."""
    from eagle_speculative_decoding_draft_gb300.engine import EagleTree
    rng = np.random.default_rng(V)
    B, d, k, m = 16, 4, 3, 9
    n = m + 1
    w = synth.custom(32, V, B, d, k, m, dtype="bf16")
    inp = synth.make_inputs(w, seed=V + 1)
    g = lambda t: t.to(dev).contiguous()
    eng = EagleTree(g(inp.w_fc), g(inp.b_fc), g(inp.w_lm), g(inp.emb), B, d, k, m)
    tree = eng.draft(g(inp.root_feat), g(inp.root_tok))
    tok, par = to_np(tree["tokens"]), to_np(tree["parents"])
    T = (rng.standard_normal((B, n, V)) * 0.05).astype(np.float32)  # coarse bf16 grid: many ties
    for b in range(B):
        for i in range(n):
            kids = np.nonzero(par[b] == i)[0]
            if kids.size and rng.random() < 0.8:
                T[b, i, tok[b, rng.choice(kids)]] = 0.25  # ties with any other 0.25 in the row
                T[b, i, rng.integers(0, V)] = 0.25
    Tb = torch.from_numpy(T).to(torch.bfloat16)
    ver = eng.verify_greedy(tree["tokens"], tree["parents"], g(Tb))
    torch.cuda.synchronize()
    ref = oracle.verify_greedy(tok, par, Tb.float().numpy(), d)
    assert np.array_equal(to_np(ver["accept_len"]), ref["accept_len"])
    assert np.array_equal(to_np(ver["accept_nodes"]), ref["accept_nodes"])
    assert np.array_equal(to_np(ver["accept_tokens"]), ref["accept_tok"])
    eng.status()
    eng.close()
