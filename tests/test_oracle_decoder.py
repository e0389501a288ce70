"""Pins of the oracle's draft decoder layer (orc_decoder_layer): one Llama decoder layer over a
tree with attention to a KV cache ("在 SGLang 里": fc, one Llama decoder layer with an identity
input norm, no final norm; chapter 04 notes §12.5: a node attends to its ancestors only).

Checked against what does not share the oracle's code: torch's float64 scaled_dot_product_attention
with an explicit mask, RoPE's relative-position property, closed forms (zero projections, a lone
node), the equality of grouped-query attention with multi-head attention on repeated key/value
weights, and the independence of a node's output from nodes outside its ancestry.
"""
import numpy as np
import pytest
import torch

import oracle
from decoder_ref import layer, reference_layer, tolerance, tree_mask

torch.manual_seed(0)


PARENTS = [-1, 0, 0, 1, 1]
DEPTHS = [0, 1, 1, 2, 2]


def run(w, d, parents=PARENTS, pos=None, new_kv=False):
    B, n, P = d["B"], d["n"], d["P"]
    mask = np.stack([tree_mask(parents)] * B)
    if pos is None:
        pos = np.array([[P + dep for dep in DEPTHS[:n]]] * B, np.int32)
    return oracle.decoder_layer(w["x"], w["w_qkv"], w["w_o"], w["w_norm"], w["w_gu"], w["w_d"], w["k_cache"],
                                w["v_cache"], pos, mask, d["H"], d["Hk"], new_kv=new_kv)


def reference_at(w, d, parents=PARENTS, pos=None):
    B, n, P = d["B"], d["n"], d["P"]
    if pos is None:
        pos = np.array([[P + dep for dep in DEPTHS[:n]]] * B, np.int32)
    return reference_layer(w, d, parents, pos)


def test_layer_within_bf16_tolerance_of_a_float64_restatement():
    """First-order bound of the bf16 rounding points: the residual sums (|h1|, |out|) and, through
    the output and down projections, the rounded attention output and MLP activations (the sums of
    absolute terms of those projections, from the float64 restatement)."""
    for seed in range(3):
        w, d = layer(seed=seed)
        got = run(w, d)["out"]
        ref, h1, absterms = reference_at(w, d)
        bound = tolerance(h1, ref, absterms)
        assert np.all(np.abs(got - ref) <= bound), np.max(np.abs(got - ref) - bound)


def test_zero_projections_leave_the_input():
    w, d = layer()
    w["w_o"] = torch.zeros_like(w["w_o"])
    w["w_d"] = torch.zeros_like(w["w_d"])
    got = run(w, d)["out"]
    assert np.array_equal(got, w["x"].float().numpy())


def test_a_lone_node_without_prefix_attends_to_itself():
    """softmax over one key: the attention output is the node's own value."""
    w, d = layer(B=1, n=1, P=0, H=2, Hk=2)
    w["w_o"] = torch.eye(d["h"], d["H"] * d["D"]).to(torch.bfloat16)  # o lands in h1's first H*D entries
    w["w_d"] = torch.zeros_like(w["w_d"])
    got = run(w, d, parents=[-1], pos=np.array([[7]], np.int32), new_kv=True)
    v = got["v_new"][0, 0].reshape(-1)  # Hk = H: v of head hq is kv head hq
    h1 = got["out"][0, 0]
    x = w["x"].float().numpy()[0, 0]
    HD = d["H"] * d["D"]
    expect = (torch.tensor(x[:HD]) + torch.tensor(v)).to(torch.bfloat16).float().numpy()
    assert np.array_equal(h1[:HD], expect)


def test_rope_depends_on_relative_position_only():
    w, d = layer(B=1, n=2, P=0, H=1, Hk=1, D=32)
    dots = []
    for shift in (0, 5, 40):
        r = run(w, d, parents=[-1, 0], pos=np.array([[3 + shift, 4 + shift]], np.int32), new_kv=True)
        k = r["k_new"][0, :, 0]
        dots.append(float(np.dot(k[0].astype(np.float64), k[1].astype(np.float64))))
    assert max(dots) - min(dots) < 2e-2 * (abs(dots[0]) + 1)


def test_grouped_query_attention_equals_repeated_multi_head():
    w, d = layer(H=4, Hk=2)
    H, Hk, D = d["H"], d["Hk"], d["D"]
    q, k, v = w["w_qkv"][:H * D], w["w_qkv"][H * D:(H + Hk) * D], w["w_qkv"][(H + Hk) * D:]
    rep = lambda t: t.reshape(Hk, D, -1).repeat_interleave(H // Hk, dim=0).reshape(H * D, -1)
    w2 = dict(w)
    w2["w_qkv"] = torch.cat([q, rep(k), rep(v)])
    kc = w["k_cache"].repeat_interleave(H // Hk, dim=2)
    vc = w["v_cache"].repeat_interleave(H // Hk, dim=2)
    w2["k_cache"], w2["v_cache"] = kc.contiguous(), vc.contiguous()
    d2 = dict(d, Hk=H)
    assert np.array_equal(run(w, d)["out"], run(w2, d2)["out"])


def test_a_node_ignores_nodes_outside_its_ancestry():
    w, d = layer()
    base = run(w, d)["out"]
    w2 = dict(w)
    x = w["x"].clone()
    x[:, 4] = x[:, 4] * -3 + 1  # node 4: a sibling of 3, not an ancestor of 0..3
    w2["x"] = x
    got = run(w2, d)["out"]
    assert np.array_equal(got[:, :4], base[:, :4])
    assert not np.array_equal(got[:, 4], base[:, 4])


def test_the_norm_epsilon_counts_for_small_activations():
    """With inputs near 1e-3 the mean square of h1 is near the epsilon (1e-6), so the epsilon
    moves the normed activation by a large factor; the output must still follow the float64
    restatement."""
    w, d = layer(seed=5)
    w["x"] = (w["x"].float() * 1e-3).to(torch.bfloat16)
    w["w_o"] = torch.zeros_like(w["w_o"])
    got = run(w, d)["out"]
    ref, h1, absterms = reference_at(w, d)
    assert np.all(np.abs(got - ref) <= tolerance(h1, ref, absterms))
