"""Pins of the oracle's greedy tree verification.

* brute force: enumerate every root path of small random trees; the accepted path is the
  longest one whose every edge carries the target's argmax at the parent, and the bonus is the
  target's argmax at its last node;
* the expected committed tokens per round E[N] = 1 + sum_i prod_{j<=i} alpha_j against the
  worked values the notes print (tests/golden/expected_tokens_per_round.json), by Monte Carlo
  over chains whose target agrees with the draft at depth i with probability alpha_i;
* the first drafted token is always accepted when the target agrees with the draft, and a
  topk = 1 chain is accepted whole.
"""
import json
from pathlib import Path

import numpy as np
import pytest

import oracle
from eagle_speculative_decoding_draft_gb300 import synth

GOLDEN = Path(__file__).resolve().parent / "golden" / "expected_tokens_per_round.json"


def random_tree(rng, n, V):
    """Parents before children; siblings get distinct tokens."""
    par = np.full(n, -1, np.int32)
    tok = np.zeros(n, np.int32)
    tok[0] = rng.integers(V)
    used = {}
    for i in range(1, n):
        p = int(rng.integers(0, i))
        par[i] = p
        taken = used.setdefault(p, set())
        t = int(rng.choice([v for v in range(V) if v not in taken]))
        taken.add(t)
        tok[i] = t
    return tok, par


def brute_force(tok, par, g):
    n = tok.shape[0]
    children = {i: [c for c in range(n) if par[c] == i] for i in range(n)}
    best = [0]

    def dfs(path):
        nonlocal best
        if len(path) > len(best):
            best = list(path)
        cur = path[-1]
        for c in children[cur]:
            if tok[c] == g[cur]:
                dfs(path + [c])

    dfs([0])
    return best


def test_verify_equals_brute_force_over_root_paths():
    rng = np.random.default_rng(2024)
    V = 6
    for trial in range(300):
        n = int(rng.integers(1, 11))
        tok, par = random_tree(rng, n, V)
        T = rng.standard_normal((n, V)).astype(np.float32)
        # plant agreements so that long accepted paths occur
        for i in range(n):
            kids = np.nonzero(par == i)[0]
            if kids.size and rng.random() < 0.7:
                T[i, tok[rng.choice(kids)]] = 10.0
        depth = 0
        for i in range(n):
            dd, a = 0, i
            while a != 0:
                a = par[a]
                dd += 1
            depth = max(depth, dd)
        out = oracle.verify_greedy(tok[None], par[None], T[None], depth)
        g = np.argmax(T, axis=1)
        path = brute_force(tok, par, g)
        L = len(path) - 1
        assert out["accept_len"][0] == L
        assert out["accept_nodes"][0, :L + 1].tolist() == path
        assert np.all(out["accept_nodes"][0, L + 1:] == -1)
        assert out["accept_tok"][0, :L].tolist() == [int(tok[c]) for c in path[1:]]
        assert out["accept_tok"][0, L] == g[path[-1]]
        assert out["g"][0].tolist() == g.tolist()


def test_target_argmax_ties_go_to_lowest_id():
    tok = np.array([[3, 1, 2]], np.int32)
    par = np.array([[-1, 0, 0]], np.int32)
    T = np.zeros((1, 3, 5), np.float32)
    T[0, 0, [1, 2]] = 1.0  # tie between tokens 1 and 2 at the root -> 1
    T[0, 1, [4, 0]] = 2.0  # tie -> 0
    out = oracle.verify_greedy(tok, par, T, 1)
    assert out["accept_len"][0] == 1
    assert out["accept_nodes"][0].tolist() == [0, 1]
    assert out["accept_tok"][0].tolist() == [1, 0]


def test_golden_values_follow_the_formula():
    for case in json.loads(GOLDEN.read_text())["cases"]:
        a = np.array(case["alpha"])
        assert round(1 + np.cumprod(a).sum(), 3) == pytest.approx(case["E_N"], abs=1e-9)


@pytest.mark.parametrize("case", json.loads(GOLDEN.read_text())["cases"],
                         ids=lambda c: str(c["E_N"]))
def test_expected_tokens_per_round_monte_carlo(case):
    alpha = np.array(case["alpha"])
    K = alpha.shape[0]
    B, V = 50_000, 4
    rng = np.random.default_rng(int(case["E_N"] * 1000))
    # chain: node i (1..K) has parent i-1 and token 1; target agrees at node i-1 w.p. alpha_i
    tok = np.tile(np.array([0] + [1] * K, np.int32), (B, 1))
    par = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    T = np.zeros((B, K + 1, V), np.float32)
    agree = rng.random((B, K)) < alpha[None, :]
    T[:, :K, 1] = np.where(agree, 1.0, 0.0)
    T[:, :K, 2] = np.where(agree, 0.0, 1.0)
    T[:, K, 3] = 1.0
    out = oracle.verify_greedy(tok, par, T, K)
    committed = out["accept_len"].astype(np.float64) + 1  # accepted drafts + the bonus token
    se = committed.std() / np.sqrt(B)
    assert abs(committed.mean() - case["E_N"]) < 4 * se + 1e-3
    assert np.all(out["accept_tok"][np.arange(B), out["accept_len"]] >= 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_first_draft_token_accepted_when_target_agrees(dtype):
    w = synth.custom(32, 400, 6, 4, 3, 9, dtype=dtype)
    inp = synth.make_inputs(w, seed=55)
    out = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok,
                            w.depth, w.topk, w.num_keep, w.is_bf16, node_logits=True)
    v = oracle.verify_greedy(out["tree_tok"], out["tree_parent"], out["node_z"], w.depth)
    assert np.all(v["accept_len"] >= 1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chain_accepted_whole_when_target_agrees(dtype):
    w = synth.custom(32, 300, 4, 5, 1, 5, dtype=dtype)
    inp = synth.make_inputs(w, seed=56)
    out = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok,
                            w.depth, w.topk, w.num_keep, w.is_bf16, node_logits=True)
    v = oracle.verify_greedy(out["tree_tok"], out["tree_parent"], out["node_z"], w.depth)
    assert np.all(v["accept_len"] == w.depth)
