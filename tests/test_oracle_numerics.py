"""Pins of the oracle's numeric building blocks against closed forms and library routines.

Each test checks the oracle against something other than itself: torch's float -> bf16
conversion, float64 matrix products within the fp32 dot-product error bound, float64
logsumexp, a full sort, and special cases with exact answers.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle

U32 = 2.0 ** -24  # unit roundoff of fp32
U_BF16 = 2.0 ** -8  # unit roundoff of bf16 (8 significant bits)


def gamma(n):
    return n * U32 / (1 - n * U32)


def torch_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x_f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F80C000,
                        0x7F7FFFFF, 0x7F7F8000, 0xFF7FFFFF, 0x00000001, 0x00008000, 0x00018000,
                        0x007FFFFF, 0x7F800000, 0xFF800000, 0x3FFF8000], dtype=np.uint32)
    bits = np.concatenate([bits, special])
    x = bits.view(np.float32)
    ours = oracle.round_bf16(x)
    ref = torch_bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN
    assert np.all(np.isnan(oracle.bf16_to_f32(ours[nan])))


def test_bf16_widening_matches_torch():
    bits = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def _rand_inputs(rng, h, V, is_bf16):
    def draw(shape, std):
        a = (rng.standard_normal(shape) * std).astype(np.float32)
        return torch_bf16_bits(a) if is_bf16 else a
    w_fc = draw((h, 2 * h), 1 / np.sqrt(2 * h))
    b_fc = draw((h,), 0.3)
    w_lm = draw((V, h), 3 / np.sqrt(h))
    emb = draw((V, h), 0.5)
    feat = (rng.standard_normal(h)).astype(np.float32)
    if is_bf16:
        feat = oracle.bf16_to_f32(torch_bf16_bits(feat))
    return w_fc, b_fc, w_lm, emb, feat


def _f64(a, is_bf16):
    return (oracle.bf16_to_f32(a) if is_bf16 else a).astype(np.float64)


@pytest.mark.parametrize("is_bf16", [False, True])
def test_fc_row_against_float64_within_dot_product_bound(is_bf16):
    rng = np.random.default_rng(11)
    h, V = 96, 40
    w_fc, b_fc, _, emb, feat = _rand_inputs(rng, h, V, is_bf16)
    tok = 17
    got = oracle.fc_row(w_fc, b_fc, feat, emb, tok, is_bf16).astype(np.float64)
    W = _f64(w_fc, is_bf16)
    x = np.concatenate([feat.astype(np.float64), _f64(emb, is_bf16)[tok]])
    b = _f64(b_fc, is_bf16)
    exact = W @ x + b
    bound = gamma(2 * h + 1) * (np.abs(W) @ np.abs(x) + np.abs(b))
    if is_bf16:
        bound = bound + U_BF16 * (np.abs(exact) + bound)
    assert np.all(np.abs(got - exact) <= bound * 1.0001 + 1e-30)
    if is_bf16:  # the output is a bf16 value
        g32 = got.astype(np.float32)
        assert np.array_equal(oracle.bf16_to_f32(torch_bf16_bits(g32)), g32)


@pytest.mark.parametrize("is_bf16", [False, True])
def test_fc_row_special_cases_select_each_half(is_bf16):
    """W_fc = [I | 0] returns the feature, [0 | I] returns the token's embedding row."""
    rng = np.random.default_rng(3)
    h, V = 32, 20
    _, _, _, emb, feat = _rand_inputs(rng, h, V, is_bf16)
    eye = np.eye(h, dtype=np.float32)
    zero = np.zeros((h, h), np.float32)
    left = np.concatenate([eye, zero], axis=1)
    right = np.concatenate([zero, eye], axis=1)
    if is_bf16:
        left, right = torch_bf16_bits(left), torch_bf16_bits(right)
    got_f = oracle.fc_row(left, None, feat, emb, 5, is_bf16)
    got_e = oracle.fc_row(right, None, feat, emb, 5, is_bf16)
    assert np.array_equal(got_f, feat)
    assert np.array_equal(got_e, _f64(emb, is_bf16)[5].astype(np.float32))


@pytest.mark.parametrize("is_bf16", [False, True])
def test_lm_head_row_against_float64_within_dot_product_bound(is_bf16):
    rng = np.random.default_rng(12)
    h, V = 128, 300
    _, _, w_lm, _, feat = _rand_inputs(rng, h, V, is_bf16)
    got = oracle.lm_head_row(w_lm, feat, is_bf16).astype(np.float64)
    W = _f64(w_lm, is_bf16)
    f = feat.astype(np.float64)
    exact = W @ f
    bound = gamma(h) * (np.abs(W) @ np.abs(f))
    assert np.all(np.abs(got - exact) <= bound * 1.0001 + 1e-30)


def test_lm_head_row_one_hot_rows_select_feature_entries():
    h, V = 16, 48
    W = np.zeros((V, h), np.float32)
    W[np.arange(V), np.arange(V) % h] = 1.0
    f = np.arange(h, dtype=np.float32) * 0.5 - 3
    z = oracle.lm_head_row(W, f, False)
    assert np.array_equal(z, f[np.arange(V) % h])


def _lse_bound(z, lse64):
    V = z.shape[0]
    # fp32 sequential sum of V terms each within one ulp of exp, then log and one add
    return (gamma(V) + 4 * U32) + 4 * U32 * abs(lse64) + 1e-7


def test_log_softmax_against_float64_logsumexp():
    rng = np.random.default_rng(5)
    for V, scale in [(1, 1.0), (7, 3.0), (1000, 2.1), (32000, 2.1), (5000, 40.0)]:
        z = (rng.standard_normal(V) * scale).astype(np.float32)
        k = min(V, 6)
        ids, logp, lse = oracle.log_softmax_topk(z, k)
        lse64 = logsumexp(z.astype(np.float64))
        assert abs(lse - lse64) <= _lse_bound(z, lse64)
        ref_logp = z[ids].astype(np.float64) - lse64
        assert np.all(np.abs(logp - ref_logp) <= _lse_bound(z, lse64) + 4 * U32 * np.abs(ref_logp))


def test_topk_is_a_full_sort_prefix_with_ties_to_lowest_id():
    rng = np.random.default_rng(9)
    for V, k in [(10, 10), (64, 5), (1000, 10), (2000, 1)]:
        z = rng.integers(-5, 6, size=V).astype(np.float32) * 0.25  # many exact ties
        ids, _, _ = oracle.log_softmax_topk(z, k)
        ref = sorted(range(V), key=lambda v: (-z[v], v))[:k]
        assert list(ids) == ref


def test_logp_of_whole_vocabulary_sums_to_one():
    rng = np.random.default_rng(21)
    V = 12
    z = (rng.standard_normal(V) * 2).astype(np.float32)
    ids, logp, lse = oracle.log_softmax_topk(z, V)
    assert sorted(ids.tolist()) == list(range(V))
    assert abs(np.exp(logp.astype(np.float64)).sum() - 1.0) < 1e-5
    assert np.all(logp <= 0)
