"""GPU sampling tree verification (eagle_verify_sample) against the oracle.

The kernel evaluates in fp32, the oracle in double precision: a decision can differ only where a
uniform falls within rounding of its threshold.  A request whose GPU result differs from the
oracle's is accepted only if the oracle reproduces it with that request's uniforms moved by
+-1e-4, and such requests must stay rare.
"""
import json
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from parity import to_np

pytestmark = pytest.mark.gpu
GOLDEN = Path(__file__).resolve().parent / "golden" / "verify_sample_cases.json"


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    return torch.device("cuda", 0)


def gpu_sample(dev, tok, par, T, Z, depth, temp, ua, ub, mode=0, threshold=0.0):
    from eagle_speculative_decoding_draft_gb300.engine import verify_sample
    g = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(dev)
    out = verify_sample(g(tok, np.int32), g(par, np.int32), g(T, np.float32), g(Z, np.float32), depth,
                        temp, g(ua, np.float32), g(ub, np.float32), mode=mode, threshold=threshold)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in out.items()}


def same(a, b, i):
    return (a["accept_len"][i] == b["accept_len"][i]
            and np.array_equal(a["accept_nodes"][i], b["accept_nodes"][i])
            and np.array_equal(a["accept_tokens" if "accept_tokens" in a else "accept_tok"][i],
                               b["accept_tokens" if "accept_tokens" in b else "accept_tok"][i]))


def as_oracle_keys(g):
    return {"accept_len": g["accept_len"], "accept_nodes": g["accept_nodes"], "accept_tok": g["accept_tokens"]}


def compare(tok, par, T, Z, depth, temp, ua, ub, got, mode=0, threshold=0.0, delta=1e-4):
    ref = oracle.verify_sample(tok, par, T, Z, depth, temp, ua, ub, mode=mode, threshold=threshold)
    g = as_oracle_keys(got)
    near = 0
    for b in range(tok.shape[0]):
        if same(g, ref, b):
            continue
        ok = False
        for d in (delta, -delta):
            ua2 = np.clip(ua[b:b + 1] + d, 0.0, 0.9999999).astype(np.float32)
            ub2 = np.clip(ub[b:b + 1] + d, 0.0, 0.9999999).astype(np.float32)
            r2 = oracle.verify_sample(tok[b:b + 1], par[b:b + 1], T[b:b + 1], Z[b:b + 1], depth, temp,
                                      ua2, ub2, mode=mode, threshold=threshold)
            one = {k: v[b:b + 1] for k, v in g.items()}
            if same(one, r2, 0):
                ok = True
                break
        assert ok, (b, {k: v[b] for k, v in g.items()}, {k: v[b] for k, v in ref.items()})
        near += 1
    return near


@pytest.mark.parametrize("case", json.loads(GOLDEN.read_text())["cases"], ids=lambda c: c["name"])
def test_worked_examples_on_the_gpu(dev, case):
    T = np.log(np.asarray(case["p"], np.float64)).astype(np.float32)[None]
    Z = np.log(np.asarray(case["q"], np.float64)).astype(np.float32)[None]
    got = gpu_sample(dev, np.array([case["tokens"]]), np.array([case["parents"]]), T, Z, case["depth"], 1.0,
                     np.array([case["u_acc"]]), np.array([case["u_bonus"]]), mode=case["mode"],
                     threshold=case["threshold"])
    assert got["accept_len"][0] == case["accept_len"]
    assert got["accept_nodes"][0].tolist() == case["accept_nodes"]
    assert got["accept_tokens"][0].tolist() == case["accept_tok"]


def random_forest(rng, B, n, k_max, V):
    """B trees of n nodes: parents precede children, siblings carry distinct tokens."""
    tok = np.zeros((B, n), np.int32)
    par = np.zeros((B, n), np.int32)
    depth = 0
    for b in range(B):
        used = [set() for _ in range(n)]
        dep = [0] * n
        par[b, 0] = -1
        tok[b, 0] = rng.integers(V)
        for i in range(1, n):
            while True:
                p = int(rng.integers(i))
                if len(used[p]) < min(k_max, V):
                    break
            t = int(rng.integers(V))
            while t in used[p]:
                t = int(rng.integers(V))
            used[p].add(t)
            par[b, i], tok[b, i] = p, t
            dep[i] = dep[p] + 1
        depth = max(depth, max(dep))
    return tok, par, depth


@pytest.mark.parametrize("B,n,V,temp,mode", [(8, 12, 100, 1.0, 0), (6, 40, 1000, 0.7, 0),
                                             (4, 61, 32000, 1.0, 0), (3, 30, 5000, 2.0, 1),
                                             (16, 5, 17, 1.0, 0), (2, 65, 128256, 1.0, 0),
                                             (5, 9, 2049, 1.3, 1),
                                             (1, 4097, 64, 1.0, 0)])  # the largest tree the call takes
def test_random_trees_match_the_oracle(dev, B, n, V, temp, mode, parity_record):
    rng = np.random.default_rng(B * 1000 + n * 10 + V)
    tok, par, depth = random_forest(rng, B, n, 4, V)
    # target close to the draft so that children are often accepted and walks go deep
    Z = (rng.standard_normal((B, n, V)) * 2.5).astype(np.float32)
    T = (Z + rng.standard_normal((B, n, V)).astype(np.float32) * 0.8).astype(np.float32)
    # draft the children where the draft is confident: put each child's token near the top of
    # its parent's draft row
    for b in range(B):
        for c in range(1, n):
            Z[b, par[b, c], tok[b, c]] += 4.0
            T[b, par[b, c], tok[b, c]] += 3.0
    ua = rng.random((B, n), dtype=np.float32)
    ub = rng.random(B, dtype=np.float32)
    thr = 0.05 if mode == 1 else 0.0
    compared, excused = 0, 0
    for d in sorted({depth, max(depth - 1, 0), 1}):
        got = gpu_sample(dev, tok, par, T, Z, d, temp, ua, ub, mode=mode, threshold=thr)
        near = compare(tok, par, T, Z, d, temp, ua, ub, got, mode=mode, threshold=thr)
        compared += B
        excused += near
        assert near <= max(1, B // 8)
    # the observed count, not only the cap: requests whose result the oracle reproduces only with
    # that request's uniforms moved by 1e-4 (fp32 kernel against the double-precision oracle)
    parity_record[f"sampling verify B{B} n{n} V{V} t{temp} mode{mode}"] = {
        "requests_compared": compared, "excused_by_uniform_shift": excused}
    print(f"sampling verify B{B} n{n} V{V}: {excused} of {compared} requests excused by a 1e-4 uniform shift")


def test_edge_cases(dev):
    rng = np.random.default_rng(1)
    V = 50
    # a root alone: only the bonus
    T = rng.standard_normal((3, 1, V)).astype(np.float32)
    ua = np.zeros((3, 1), np.float32)
    ub = np.array([0.0, 0.5, 0.9999], np.float32)
    got = gpu_sample(dev, np.zeros((3, 1), np.int32), -np.ones((3, 1), np.int32), T, T, 3, 1.0, ua, ub)
    compare(np.zeros((3, 1), np.int32), -np.ones((3, 1), np.int32), T, T, 3, 1.0, ua, ub, got)
    assert got["accept_len"].tolist() == [0, 0, 0]
    assert (got["accept_nodes"][:, 1:] == -1).all()
    # depth 0: children are never tested
    tok, par, _ = random_forest(rng, 4, 10, 3, V)
    T = rng.standard_normal((4, 10, V)).astype(np.float32)
    got = gpu_sample(dev, tok, par, T, T, 0, 1.0, np.zeros((4, 10), np.float32), np.full(4, 0.3, np.float32))
    assert got["accept_len"].tolist() == [0] * 4
    # out-of-range child tokens are never accepted
    tok2 = tok.copy()
    tok2[:, 1:] = V + 5
    got = gpu_sample(dev, tok2, par, T, T, 5, 1.0, np.zeros((4, 10), np.float32), np.full(4, 0.3, np.float32))
    assert got["accept_len"].tolist() == [0] * 4
    # an empty batch launches nothing
    from eagle_speculative_decoding_draft_gb300 import _lib
    lib = _lib.load()
    assert lib.eagle_verify_sample(0, 1, V, 1, *([None] * 4), 1.0, 0, 0.0, *([None] * 6), None) == 0


def test_lossless_on_the_gpu(dev):
    """Children drawn from q: the first emitted token is distributed as p (chi-square)."""
    rng = np.random.default_rng(21)
    V, k, N = 7, 3, 40000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    n = 1 + k
    tok = np.zeros((N, n), np.int32)
    tok[:, 1:] = rng.choice(V, size=(N, k), p=q)
    par = np.tile(np.array([-1] + [0] * k, np.int32), (N, 1))
    T = np.tile(np.log(p).astype(np.float32), (N, n, 1))
    Z = np.tile(np.log(q).astype(np.float32), (N, n, 1))
    ua = rng.random((N, n), dtype=np.float32)
    ub = rng.random(N, dtype=np.float32)
    got = gpu_sample(dev, tok, par, T, Z, 1, 1.0, ua, ub)
    counts = np.bincount(got["accept_tokens"][:, 0], minlength=V)
    chi2 = float(np.sum((counts - N * p) ** 2 / (N * p)))
    assert chi2 < 40.0, (chi2, counts, N * p)  # 6 dof
