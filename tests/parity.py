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


def _window(info, mg, thr):
    """Counts one compared decision by the window its margin falls in."""
    info["decisions"] += 1
    if mg <= MARGIN:
        info["within_1e3"] += 1
    elif mg <= thr:
        info["widened_only"] += 1


def lockstep_compare(ref, j, gpu, b, k, d, m, is_bf16):
    """Walks request b (oracle request j) level by level while both sides expand the same nodes.

    gpu: dict with "logits" [d][R][V] (numpy-convertible per row), "pool_tok", "pool_S",
    "pool_parent" [B][n_cand].  While the rows agree their logits must be within tolerance.  A
    decision (a row's top-k children, a frontier, the rerank cut) may differ only if its margin in
    the oracle's values is at most max(MARGIN, 2 * deviation), where deviation is the largest
    GPU-oracle difference of the values it compares, measured at that level.  Returns a dict:
    exact (bool), level of divergence, margin, threshold, the per-level max |dz|, and counts of
    the decisions compared: all, those with margin <= 1e-3, and those whose margin lies above
    1e-3 but within the widened threshold (a divergence there is excused only by the widening)."""
    info = {"exact": False, "diverged_at": None, "margin": None, "threshold": None, "dz": [],
            "decisions": 0, "within_1e3": 0, "widened_only": 0}
    e_S = 0.0
    for l in range(d):
        base = 0 if l == 0 else k + (l - 1) * k * k
        nl = k if l == 0 else k * k
        if l >= 2:
            pb = k + (l - 2) * k * k
            mg = float(np.min(top_gaps(ref["cand_S"][j, pb:pb + k * k], k + 1)))
            thr = max(MARGIN, 2 * e_S)
            _window(info, mg, thr)
        if l >= 1:
            g_front = [int(gpu["pool_parent"][b, base + s * k]) for s in range(k)]
            o_front = ref["front_cand"][l][j].tolist()
            if g_front != o_front:
                # level 1's frontier is every child of the root in child order: it cannot differ
                # unless the root's children did, which is checked (and returned) below
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
            mg = float(np.min(top_gaps(ref["row_z"][l, ro], k + 1)))
            thr = max(MARGIN, 2 * e_z)
            _window(info, mg, thr)
            if not np.array_equal(gpu["pool_tok"][b, c0:c0 + k], ref["cand_tok"][j, c0:c0 + k]):
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
    if 0 < m < nc:
        srt = np.sort(ref["cand_S"][j])[::-1]
        mg = float(srt[m - 1] - srt[m])
        e_all = float(np.max(np.abs(gpu["pool_S"][b].astype(np.float64) - ref["cand_S"][j])))
        thr = max(MARGIN, 2 * e_all)
        _window(info, mg, thr)
        g_keep = set(np.argsort(-gpu["pool_S"][b], kind="stable")[:m].tolist())
        o_keep = set(np.argsort(-ref["cand_S"][j], kind="stable")[:m].tolist())
        if g_keep != o_keep:
            assert mg <= thr, f"request {b}: rerank cut differs with margin {mg:.3g} above {thr:.3g}"
            info.update(diverged_at=d, margin=mg, threshold=thr)
            return info
    info["exact"] = True
    return info


def bf16_ulp(x):
    """One bf16 unit in the last place at |x| (the spacing of bf16 numbers there)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def tree_from_pool(pool_tok, pool_S, pool_parent, root_tok, k, m, pos_base):
    """The rerank and tree build written out from their definitions on one request's pool: keep
    the m best candidates by (S descending, candidate ascending); order the kept ones by
    candidate id (level-major, parents first) after the root; parent = the tree index of the
    parent candidate (the root for depth 1); position = depth + base; mask row i = i and its
    ancestors.  Returns tok, parent, pos, S, mask (bool [n][n])."""
    nc = pool_S.shape[0]
    order = sorted(range(nc), key=lambda c: (-float(pool_S[c]), c))[:m]
    kept = sorted(order)
    idx = {c: i + 1 for i, c in enumerate(kept)}
    n = m + 1
    tok = np.zeros(n, np.int64)
    par = np.full(n, -1, np.int64)
    dep = np.zeros(n, np.int64)
    S = np.zeros(n, np.float32)
    tok[0] = root_tok
    for c, i in idx.items():
        tok[i] = pool_tok[c]
        S[i] = pool_S[c]
        pc = int(pool_parent[c])
        if pc < 0:
            par[i] = 0
        else:
            assert pc in idx, f"kept candidate {c} without its parent {pc}"
            par[i] = idx[pc]
        dep[i] = dep[par[i]] + 1
    mask = np.eye(n, dtype=bool)
    for i in range(1, n):
        mask[i] |= mask[par[i]]
    return tok, par, dep + pos_base, S, mask


def teacher_forced_check(inp, w, gpu, b, logits_rows, T_b, ver_b, pos_base, rec):
    """Checks request b of a GPU step level by level against the oracle fed the GPU's own inputs.

    Every draft row's input [f^ of the row that produced its node || E[token]] is taken from the
    GPU's intermediate state, so each comparison sees one level's arithmetic only (no drift
    carried from earlier levels), and the parity rule applies as written: a decision may differ
    only where its margin is at most 1e-3.  Checked per row: f^ against the oracle's FC (equal
    up to one bf16 rounding step, i.e. one ulp, in at most 1% of the elements), the logits against
    the oracle's LM head on the GPU's f^ (2e-2 absolute for bf16, 1e-4 relative for fp32), the top-k
    children against the oracle's top-k of those logits, and each child's score against
    fl(S(parent) + logp).  Then exactly: the next frontier (top-k of the level's children by
    (S desc, candidate asc)), the rerank/build of the GPU pool, and greedy verification of the
    GPU tree against the oracle's walk.

    gpu: numpy arrays fhat [d][r_pad][h] (float32), pool_tok / pool_S / pool_parent / pool_row
    [B][n_cand], and the built tree tokens / parents / positions / mask / logscore [B][...].
    logits_rows(l, r) returns the GPU logits of row r at level l; T_b [n][V] the request's target
    logits; ver_b (accept_len, accept_nodes, accept_tokens) the GPU's verify result."""
    import oracle
    k, d, m, h = w.topk, w.depth, w.num_keep, w.hidden
    is_bf16 = w.is_bf16
    feat0 = (inp.root_feat[b].float() if hasattr(inp.root_feat, "float") else inp.root_feat[b])
    feat0 = np.asarray(feat0, np.float32)
    tok0 = int(inp.root_tok[b])
    nc = w.num_candidates
    same_tree = True  # no decision of the request differs from the oracle's on the same inputs
    P = gpu["pool_tok"][b], gpu["pool_S"][b], gpu["pool_parent"][b], gpu["pool_row"][b]
    ptok, pS, ppar, prow = P
    for l in range(d):
        base = 0 if l == 0 else k + (l - 1) * k * k
        nrows = 1 if l == 0 else k
        for s in range(nrows):
            row = b if l == 0 else b * k + s
            c0 = base + s * k
            if l == 0:
                feat, tok, S_par = feat0, tok0, np.float32(0.0)
            else:
                pc = int(ppar[c0])
                assert all(int(ppar[c0 + j]) == pc for j in range(k)), "children of one row disagree on the parent"
                lp = 0 if pc < k else 1 + (pc - k) // (k * k)
                feat = gpu["fhat"][lp, int(prow[pc])]
                tok, S_par = int(ptok[pc]), np.float32(pS[pc])
            fo = oracle.fc_row(inp.w_fc, inp.b_fc, feat, inp.emb, tok, is_bf16)
            fg = gpu["fhat"][l, row]
            diff = fg != fo
            rec["fhat_elems"] += h
            if is_bf16:
                nflip = int(np.count_nonzero(diff))
                rec["fhat_flips"] += nflip
                if nflip:
                    # both sides round their own fp32 sum, each within gamma_2h sum|w x| of the
                    # exact value, to bf16: they may differ by that bound plus one bf16 step
                    x = np.concatenate([np.asarray(feat, np.float32), emb_row(inp, tok)])
                    absdot = fc_absdot(inp, x)[diff] + np.abs(bias_f32(inp)[diff])
                    bound = 2 * gamma32(2 * h + 1) * absdot + bf16_ulp(np.maximum(np.abs(fg[diff]), np.abs(fo[diff])))
                    gap = np.abs(fg[diff].astype(np.float64) - fo[diff])
                    assert np.all(gap <= bound), (f"level {l} row {row}: f^ differs beyond the fp32 bound "
                                                  f"plus one bf16 step: {gap[gap > bound][:4]} > {bound[gap > bound][:4]}")
                assert nflip <= max(2, h // 100), f"level {l} row {row}: {nflip} f^ elements differ"
            else:
                assert np.all(np.abs(fg - fo) <= F32_REL * np.maximum(1.0, np.abs(fo))), f"level {l} row {row}: f^"
            zo = oracle.lm_head_row(inp.w_lm, fg, is_bf16)
            zg = np.asarray(logits_rows(l, row), np.float32)
            assert_close_logits(zg, zo, is_bf16, f"teacher-forced level {l} row {row}")
            rec["max_dz"] = max(rec["max_dz"], float(np.max(np.abs(zg.astype(np.float64) - zo))))
            ids_o, logp_o, _ = oracle.log_softmax_topk(zo, k)
            mg = float(np.min(top_gaps(zo, k + 1)))
            rec["rows"] += 1
            if mg <= MARGIN:
                rec["rows_within_1e3"] += 1
            ids_g = ptok[c0:c0 + k]
            if not np.array_equal(ids_g, ids_o):
                assert mg <= MARGIN, (f"level {l} row {row}: top-{k} differs from the oracle's with "
                                      f"margin {mg:.3g} > {MARGIN}")
                rec["rows_diverged"] += 1
                same_tree = False
            same = ids_g == ids_o
            S_o = (S_par + logp_o.astype(np.float32)).astype(np.float32)
            assert_close_logits(pS[c0:c0 + k][same], S_o[same], is_bf16, f"level {l} row {row}: scores")
        # the next frontier, exactly, from the GPU's own scores
        if l < d - 1:
            nxt = k + l * k * k
            got = [int(ppar[nxt + s * k]) for s in range(k)]
            if l == 0:
                want = list(range(k))
            else:
                want = sorted(range(base, base + k * k), key=lambda c: (-float(pS[c]), c))[:k]
            assert got == want, f"level {l + 1} frontier {got} != {want}"
    tok, par, pos, S, mask = tree_from_pool(ptok, pS, ppar, tok0, k, m, pos_base)
    n = m + 1
    assert np.array_equal(gpu["tokens"][b], tok)
    assert np.array_equal(gpu["parents"][b], par)
    assert np.array_equal(gpu["positions"][b], pos)
    assert np.array_equal(unpack_mask(gpu["mask"][b], n), mask)
    assert np.array_equal(gpu["logscore"][b].astype(np.float32), S)
    ref = oracle.verify_greedy(gpu["tokens"][b:b + 1], gpu["parents"][b:b + 1], T_b[None], d)
    assert ver_b[0] == ref["accept_len"][0]
    assert np.array_equal(ver_b[1], ref["accept_nodes"][0])
    assert np.array_equal(ver_b[2], ref["accept_tok"][0])
    rec["requests"] += 1
    rec["exact_trees"] += int(same_tree)


def gamma32(n):
    """n u / (1 - n u) for fp32 (u = 2^-24): the relative bound of an n-term fp32 sum."""
    u = 2.0 ** -24
    return n * u / (1 - n * u)


_ABS_W = {"w": None, "abs": None}


def fc_absdot(inp, x):
    """sum_i |W_fc[o][i]| |x_i| for every output o (float64), |W_fc| kept for the last weight
    tensor seen (held by reference, so a new tensor at a reused address is not mistaken for it)."""
    if _ABS_W["w"] is not inp.w_fc:
        _ABS_W["w"] = inp.w_fc
        _ABS_W["abs"] = np.abs(inp.w_fc.float().numpy()).astype(np.float32)
    return (_ABS_W["abs"] @ np.abs(x).astype(np.float32)).astype(np.float64) * (1 + 1e-6)


def emb_row(inp, tok):
    return inp.emb[int(tok)].float().numpy().astype(np.float32)


def bias_f32(inp):
    return inp.b_fc.float().numpy().astype(np.float64)


def new_tf_record():
    return {"requests": 0, "exact_trees": 0, "rows": 0, "rows_within_1e3": 0, "rows_diverged": 0,
            "fhat_elems": 0, "fhat_flips": 0, "max_dz": 0.0}


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
