"""Helpers shared by the GPU parity tests: tolerances, decision margins, tree comparison.

Tolerances: logits and log-probabilities within 2e-2 absolute for bf16 configurations and 1e-4
relative for fp32 (read as |d| <= 1e-4 * max(1, |ref|)).  Integer decisions (children, frontier,
rerank cut) must agree unless their margin in the oracle's values is at most
max(1e-3, 2 * the GPU-oracle deviation measured at that level).  The deviation is not a fixed
number because the FC output is rounded to bf16 and fed to the next level: a one-ulp rounding
disagreement at level 0 (fp32 summation order) grows level by level, for any two fp32
evaluation orders (CPU fp32 against CPU float64 drifts the same way).  Where every decision
agrees, the tree arrays, mask, positions and the verify result must be bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

MARGIN = 1e-3
BF16_ABS = 2e-2
F32_REL = 1e-4


def close_logits(got, ref, is_bf16):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if is_bf16:
        return np.abs(got - ref) <= BF16_ABS
    return np.abs(got - ref) <= F32_REL * np.maximum(1.0, np.abs(ref))


def assert_close_logits(got, ref, is_bf16, what=""):
    ok = close_logits(got, ref, is_bf16)
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {np.count_nonzero(~ok)} values out of tolerance, first at "
                             f"{tuple(i)}: got {np.asarray(got)[tuple(i)]} ref {np.asarray(ref)[tuple(i)]}")


def request_rows(b, k, d):
    """(level, row) of every draft row of request b."""
    return [(0, b)] + [(l, b * k + s) for l in range(1, d) for s in range(k)]


def top_gaps(values, count):
    """Gaps between consecutive entries of the `count` largest values (descending)."""
    top = np.sort(np.asarray(values, np.float64))[::-1][:count]
    return top[:-1] - top[1:] if top.shape[0] > 1 else np.array([np.inf])


def lockstep_compare(ref, j, gpu, b, k, d, m, is_bf16):
    """Walks request b (oracle request j) level by level while both sides expand the same nodes.

    gpu: dict with "logits" [d][R][V] (numpy-convertible per row), "pool_tok", "pool_S",
    "pool_parent" [B][n_cand].  While the rows agree their logits must be within tolerance.  A
    decision (a row's top-k children, a frontier, the rerank cut) may differ only if its margin in
    the oracle's values is at most max(MARGIN, 2 * deviation), where deviation is the largest
    GPU-oracle difference of the values it compares, measured at that level.  Returns a dict:
    exact (bool), level of divergence, margin, threshold and the per-level max |dz|."""
    info = {"exact": False, "diverged_at": None, "margin": None, "threshold": None, "dz": []}
    e_S = 0.0
    for l in range(d):
        base = 0 if l == 0 else k + (l - 1) * k * k
        nl = k if l == 0 else k * k
        if l >= 1:
            g_front = [int(gpu["pool_parent"][b, base + s * k]) for s in range(k)]
            o_front = ref["front_cand"][l][j].tolist()
            if g_front != o_front:
                pb = k + (l - 2) * k * k if l >= 2 else 0
                pn = k if l == 1 else k * k
                mg = float(np.min(top_gaps(ref["cand_S"][j, pb:pb + pn], k + 1)))
                thr = max(MARGIN, 2 * e_S)
                assert mg <= thr, (f"request {b}: frontier of level {l} differs with margin {mg:.3g} "
                                   f"above {thr:.3g}")
                info.update(diverged_at=l, margin=mg, threshold=thr)
                return info
        rows = [(b, j)] if l == 0 else [(b * k + s, j * k + s) for s in range(k)]
        e_z = 0.0
        for rg, ro in rows:
            zg = to_np(gpu["logits"][l, rg])
            assert_close_logits(zg, ref["row_z"][l, ro], is_bf16, f"level {l} row {rg}")
            e_z = max(e_z, float(np.max(np.abs(zg.astype(np.float64) - ref["row_z"][l, ro]))))
        info["dz"].append(e_z)
        for s, (rg, ro) in enumerate(rows):
            c0 = base + s * k
            if not np.array_equal(gpu["pool_tok"][b, c0:c0 + k], ref["cand_tok"][j, c0:c0 + k]):
                mg = float(np.min(top_gaps(ref["row_z"][l, ro], k + 1)))
                thr = max(MARGIN, 2 * e_z)
                assert mg <= thr, (f"request {b}: children of level {l} row {rg} differ with "
                                   f"margin {mg:.3g} above {thr:.3g}")
                info.update(diverged_at=l, margin=mg, threshold=thr)
                return info
        e_S = float(np.max(np.abs(gpu["pool_S"][b, base:base + nl].astype(np.float64)
                                  - ref["cand_S"][j, base:base + nl])))
        if is_bf16:
            assert e_S <= BF16_ABS * (l + 1)
    # rerank cut
    nc = ref["cand_S"].shape[1]
    g_keep = set(np.argsort(-gpu["pool_S"][b], kind="stable")[:m].tolist())
    o_keep = set(np.argsort(-ref["cand_S"][j], kind="stable")[:m].tolist())
    if 0 < m < nc and g_keep != o_keep:
        mg = float(np.sort(ref["cand_S"][j])[::-1][m - 1] - np.sort(ref["cand_S"][j])[::-1][m])
        e_all = float(np.max(np.abs(gpu["pool_S"][b].astype(np.float64) - ref["cand_S"][j])))
        thr = max(MARGIN, 2 * e_all)
        assert mg <= thr, f"request {b}: rerank cut differs with margin {mg:.3g} above {thr:.3g}"
        info.update(diverged_at=d, margin=mg, threshold=thr)
        return info
    info["exact"] = True
    return info


def tree_paths(tok, par):
    out = set()
    for i in range(1, tok.shape[0]):
        p, a = [], i
        while a > 0:
            p.append(int(tok[a]))
            a = par[a]
        out.add(tuple(reversed(p)))
    return out


def unpack_mask(words, n):
    words = np.asarray(words).astype(np.uint32)
    bits = np.zeros((words.shape[0], n), dtype=bool)
    for j in range(n):
        bits[:, j] = (words[:, j // 32] >> np.uint32(j % 32)) & np.uint32(1)
    return bits


def assert_valid_tree(tok, par, pos, mask, S, depth, pos_base=0):
    """Properties every built tree has, whatever its near-tie decisions."""
    n = tok.shape[0]
    dep = np.zeros(n, int)
    assert par[0] == -1
    for i in range(1, n):
        assert 0 <= par[i] < i
        dep[i] = dep[par[i]] + 1
        assert S[i] <= S[par[i]]
    assert dep.max() <= depth
    assert np.array_equal(pos, dep + pos_base)
    closure = np.eye(n, dtype=bool)
    for i in range(1, n):
        closure[i] |= closure[par[i]]
    assert np.array_equal(unpack_mask(mask, n), closure)


def to_np(t):
    return t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
