"""The GPU parity helpers checked on the CPU: the teacher-forced comparison and the decision
windows of the free-running one accept the oracle's own step and reject planted mistakes.

The oracle's intermediate state stands in for the GPU's (same layout: f^ of every level's rows,
the rerank pool, the built tree), so these tests run without a GPU."""
import numpy as np
import pytest

import oracle
from eagle_speculative_decoding_draft_gb300 import synth
from parity import lockstep_compare, new_tf_record, teacher_forced_check, tree_from_pool


def oracle_as_gpu(w, inp, pos_base):
    ref = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, inp.root_feat, inp.root_tok,
                            w.depth, w.topk, w.num_keep, w.is_bf16, pos_base=pos_base,
                            row_logits=True, node_logits=True)
    gpu = {"fhat": ref["row_fhat"], "pool_tok": ref["cand_tok"], "pool_S": ref["cand_S"],
           "pool_parent": ref["cand_parent"], "pool_row": ref["cand_row"],
           "tokens": ref["tree_tok"], "parents": ref["tree_parent"], "positions": ref["tree_pos"],
           "mask": ref["tree_mask"].view(np.int32), "logscore": ref["tree_S"],
           "logits": ref["row_z"]}
    return ref, gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_teacher_forced_accepts_the_oracles_own_step(dtype):
    w = synth.custom(64, 300, 3, 4, 3, 12, dtype=dtype)
    inp = synth.make_inputs(w, seed=77)
    pos = np.array([5, 6, 7], np.int32)
    ref, gpu = oracle_as_gpu(w, inp, pos)
    T = ref["node_z"] + synth.target_noise(inp)
    ver = oracle.verify_greedy(ref["tree_tok"], ref["tree_parent"], T, w.depth)
    rec = new_tf_record()
    for b in range(w.batch):
        teacher_forced_check(inp, w, gpu, b, lambda l, r: ref["row_z"][l, r], T[b],
                             (ver["accept_len"][b], ver["accept_nodes"][b], ver["accept_tok"][b]),
                             int(pos[b]), rec)
    assert rec["requests"] == 3 and rec["rows"] == 3 * (1 + 3 * 3)
    assert rec["fhat_flips"] == 0 and rec["rows_diverged"] == 0 and rec["max_dz"] == 0.0
    for b in range(w.batch):
        info = lockstep_compare(ref, b, gpu, b, w.topk, w.depth, w.num_keep, w.is_bf16)
        assert info["exact"] and info["decisions"] > 0


def test_teacher_forced_rejects_planted_mistakes():
    w = synth.custom(64, 300, 2, 3, 3, 8, dtype="bf16")
    inp = synth.make_inputs(w, seed=78)
    pos = np.zeros(2, np.int32)
    ref, gpu = oracle_as_gpu(w, inp, pos)
    T = ref["node_z"] + synth.target_noise(inp)
    ver = oracle.verify_greedy(ref["tree_tok"], ref["tree_parent"], T, w.depth)
    vb = (ver["accept_len"][0], ver["accept_nodes"][0], ver["accept_tok"][0])

    def check(g, logits=None, v=vb):
        z = ref["row_z"] if logits is None else logits
        teacher_forced_check(inp, w, g, 0, lambda l, r: z[l, r], T[0], v, 0, new_tf_record())

    check(gpu)
    bad = {k: v.copy() for k, v in gpu.items()}
    bad["pool_tok"][0, [3, 4]] = bad["pool_tok"][0, [4, 3]]  # two children of level 1 swapped
    with pytest.raises(AssertionError):
        check(bad)
    bad = {k: v.copy() for k, v in gpu.items()}
    bad["fhat"][1, 0, :8] += 0.25  # an f^ row off by far more than one ulp
    with pytest.raises(AssertionError):
        check(bad)
    z = ref["row_z"].copy()
    z[1, 1, 5] += 0.1  # a logit off by more than the tolerance
    with pytest.raises(AssertionError):
        check(gpu, logits=z)
    bad = {k: v.copy() for k, v in gpu.items()}
    bad["parents"][0, -1] = 0  # a tree node re-parented
    with pytest.raises(AssertionError):
        check(bad)
    with pytest.raises(AssertionError):  # a verify result off by one accepted node
        check(gpu, v=(vb[0] + 1, vb[1], vb[2]))


def test_tree_from_pool_keeps_parents_first():
    # pool of k = 2, d = 2: candidates 0, 1 (children of the root), 2..5 (2, 3 under 0; 4, 5 under 1)
    S = np.array([-0.1, -0.5, -0.3, -0.9, -0.6, -0.7], np.float32)
    tok = np.array([10, 11, 12, 13, 14, 15])
    par = np.array([-1, -1, 0, 0, 1, 1])
    t, p, pos, s, mask = tree_from_pool(tok, S, par, 99, 2, 4, 3)
    assert t.tolist() == [99, 10, 11, 12, 14] and p.tolist() == [-1, 0, 0, 1, 2]
    assert pos.tolist() == [3, 4, 4, 5, 5]
    assert mask[4].tolist() == [True, False, True, False, True]
