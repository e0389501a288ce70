"""Pins of the oracle's sampling tree verification (orc_verify_sample).

The rule is the one of "EAGLE 推测解码为什么比 Medusa 快？" (chapter 04 notes) §6.2: a drafted
token t is accepted when r <= min(1, p(t)/q(t)); on rejection sampling continues from
norm(max(0, p - q)), child after child; §7.1: with q == p the test always passes.  The threshold
variant follows the SGLang note in the "Summary" of "(EAGLE 1) EAGLE: Speculative Sampling
Requires Rethinking Feature Uncertainty".
"""
import json
from pathlib import Path

import numpy as np
import pytest

import oracle

GOLDEN = Path(__file__).resolve().parent / "golden" / "verify_sample_cases.json"


def _logits(probs):
    return np.log(np.asarray(probs, dtype=np.float64)).astype(np.float32)


@pytest.mark.parametrize("case", json.loads(GOLDEN.read_text())["cases"], ids=lambda c: c["name"])
def test_worked_examples(case):
    T = _logits(case["p"])[None]
    Z = _logits(case["q"])[None]
    r = oracle.verify_sample([case["tokens"]], [case["parents"]], T, Z, case["depth"], 1.0,
                             [case["u_acc"]], [case["u_bonus"]], mode=case["mode"],
                             threshold=case["threshold"])
    assert r["accept_len"][0] == case["accept_len"]
    assert r["accept_nodes"][0].tolist() == case["accept_nodes"]
    assert r["accept_tok"][0].tolist() == case["accept_tok"]


def random_tree(rng, n, k_max, V):
    """Parents precede children; siblings carry distinct tokens."""
    par = [-1]
    tok = [int(rng.integers(V))]
    used = {0: set()}
    depth = {0: 0}
    for i in range(1, n):
        while True:
            p = int(rng.integers(i))
            if len(used[p]) < min(k_max, V):
                break
        t = int(rng.integers(V))
        while t in used[p]:
            t = int(rng.integers(V))
        used[p].add(t)
        used[i] = set()
        par.append(p)
        tok.append(t)
        depth[i] = depth[p] + 1
    return np.array(tok, np.int32), np.array(par, np.int32), max(depth.values())


def first_child_path(tok, par, depth_limit):
    cur, path = 0, [0]
    while len(path) - 1 < depth_limit:
        kids = [c for c in range(1, len(tok)) if par[c] == cur]
        if not kids:
            break
        cur = kids[0]
        path.append(cur)
    return path


def test_q_equal_p_accepts_the_first_child_everywhere():
    """Chapter 04 §7.1: sum_x q(x) min(1, p(x)/q(x)) = 1 when q == p."""
    rng = np.random.default_rng(7)
    for trial in range(20):
        n, V = int(rng.integers(2, 30)), int(rng.integers(8, 60))
        tok, par, d = random_tree(rng, n, 4, V)
        T = (rng.standard_normal((1, n, V)) * 2).astype(np.float32)
        ua = rng.random((1, n), dtype=np.float32) * np.float32(0.999)
        r = oracle.verify_sample(tok[None], par[None], T, T.copy(), d, 0.7, ua, [0.5])
        path = first_child_path(tok, par, d)
        assert r["accept_len"][0] == len(path) - 1
        assert r["accept_nodes"][0][:len(path)].tolist() == path


def test_lossless_when_children_are_drawn_from_q():
    """The first token emitted (an accepted child of the root, or the bonus) is distributed as
    p_root when the root's children are independent draws from q_root: SpecInfer's
    multi-candidate rejection sampling, which chapter 04 §6.2 says keeps the target distribution
    exactly.  Chi-square over many independent requests in one call."""
    rng = np.random.default_rng(11)
    V, k, N = 6, 3, 60000
    for trial in range(3):
        p = rng.dirichlet(np.ones(V) * 0.8)
        q = rng.dirichlet(np.ones(V) * 0.8)
        n = 1 + k
        tok = np.zeros((N, n), np.int32)
        tok[:, 1:] = rng.choice(V, size=(N, k), p=q)
        par = np.tile(np.array([-1] + [0] * k, np.int32), (N, 1))
        T = np.tile(np.log(p).astype(np.float32), (N, n, 1))
        Z = np.tile(np.log(q).astype(np.float32), (N, n, 1))
        ua = rng.random((N, n), dtype=np.float32)
        ub = rng.random(N, dtype=np.float32)
        r = oracle.verify_sample(tok, par, T, Z, 1, 1.0, ua, ub)
        first = r["accept_tok"][:, 0]
        counts = np.bincount(first, minlength=V)
        expected = N * p
        chi2 = float(np.sum((counts - expected) ** 2 / expected))
        assert chi2 < 35.0, (chi2, counts, expected)  # 5 dof; P(chi2 > 35) < 2e-6


def test_lossless_check_catches_a_wrong_residual():
    """The chi-square pin is sharp: drawing the bonus from p itself after a rejection (dropping
    the residual) is detected."""
    rng = np.random.default_rng(3)
    V, N = 5, 60000
    p = np.array([0.4, 0.3, 0.15, 0.1, 0.05])
    q = np.array([0.05, 0.1, 0.15, 0.3, 0.4])
    child = rng.choice(V, size=N, p=q)
    u = rng.random(N)
    ub = rng.random(N)
    cdf = np.cumsum(p)
    wrong = np.where(u <= np.minimum(1, p[child] / q[child]), child, np.searchsorted(cdf, ub, side="right"))
    counts = np.bincount(wrong, minlength=V)
    chi2 = float(np.sum((counts - N * p) ** 2 / (N * p)))
    assert chi2 > 35.0


def test_depth_limit_and_leaves_draw_the_bonus_from_p():
    rng = np.random.default_rng(5)
    V = 16
    tok = np.array([3, 4, 5], np.int32)      # chain root -> 1 -> 2
    par = np.array([-1, 0, 1], np.int32)
    T = (rng.standard_normal((1, 3, V))).astype(np.float32)
    # depth limit 1: node 1 accepted (q == p) and its child is never tested
    r = oracle.verify_sample(tok[None], par[None], T, T.copy(), 1, 1.0, [[0.0, 0.5, 0.5]], [0.0])
    assert r["accept_len"][0] == 1 and r["accept_nodes"][0].tolist() == [0, 1]
    # with u_bonus = 0 the bonus is the first token of positive probability at node 1: token 0
    assert r["accept_tok"][0].tolist() == [4, 0]


def test_threshold_limits():
    rng = np.random.default_rng(9)
    for trial in range(10):
        n, V = int(rng.integers(2, 20)), 32
        tok, par, d = random_tree(rng, n, 3, V)
        T = (rng.standard_normal((1, n, V)) * 3).astype(np.float32)
        Z = (rng.standard_normal((1, n, V)) * 3).astype(np.float32)
        ua = rng.random((1, n), dtype=np.float32)
        # threshold 0 accepts the first child at every node
        r0 = oracle.verify_sample(tok[None], par[None], T, Z, d, 1.0, ua, [0.3], mode=1, threshold=0.0)
        path = first_child_path(tok, par, d)
        assert r0["accept_nodes"][0][:len(path)].tolist() == path
        # threshold above 1 accepts nothing
        r1 = oracle.verify_sample(tok[None], par[None], T, Z, d, 1.0, ua, [0.3], mode=1, threshold=1.5)
        assert r1["accept_len"][0] == 0


def test_temperature_divides_the_logits():
    rng = np.random.default_rng(13)
    n, V = 12, 40
    tok, par, d = random_tree(rng, n, 3, V)
    T = (rng.standard_normal((1, n, V)) * 3).astype(np.float32)
    Z = (rng.standard_normal((1, n, V)) * 3).astype(np.float32)
    ua = rng.random((1, n), dtype=np.float32)
    a = oracle.verify_sample(tok[None], par[None], T, Z, d, 2.0, ua, [0.37])
    b = oracle.verify_sample(tok[None], par[None], T / 2, Z / 2, d, 1.0, ua, [0.37])
    for key in a:
        assert np.array_equal(a[key], b[key])
