"""The GEMM entry point that allocates nothing (eagle_linear_bf16_noalloc).

Some callers cannot allocate device memory (no cudaMalloc where it would synchronise the device
or where a host framework owns all memory).  For them the library keeps the GEMM's split-K
scratch in a fixed array of its own device memory.  This test calls that entry point through the
C ABI twice in a row and checks each result against the oracle's fp32 dot products and against
the allocating entry point (eagle_linear_bf16, with a scratch buffer from torch), both within the
fp32 dot-product bound used by the other GEMM tests; on a GPU with at most 160 SMs the two entry
points split the work identically, so there they must also agree bit for bit.  The shapes cover
every way the array is used: stream-K with the in-launch fix-up (10 rows), one row, few weight
tiles with a second launch summing the partials (777 x 1000 at 32 rows), and 17-32 rows over 250
weight tiles on CTA pairs, which fills the whole partials region and needs the tickets reset
between the two calls.  It also checks that oversize requests are refused.  It sits in a file
that pytest collects last and passes both alone and after the other tests.
"""
import ctypes

import numpy as np

import oracle
import pytest
import torch

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


def gamma(n):
    return n * U32 / (1 - n * U32)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from eagle_speculative_decoding_draft_gb300 import build, _lib
    build.build()
    return _lib.load()


def _noalloc(lib, w, x, bias, out_bf16):
    M, K = w.shape
    rows = x.shape[0]
    y = torch.empty(rows, M, dtype=torch.bfloat16 if out_bf16 else torch.float32, device=w.device)
    P = ctypes.c_void_p
    rc = lib.eagle_linear_bf16_noalloc(P(w.data_ptr()), w.stride(0), P(x.data_ptr()), x.stride(0),
                                       P(bias.data_ptr()), M, K, rows, P(y.data_ptr()), y.stride(0),
                                       int(out_bf16),
                                       P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.eagle_status_str(rc)
    return y


@pytest.mark.parametrize("M,K,rows,out_bf16", [(32000, 4096, 10, False), (4096, 8192, 1, True),
                                               (777, 1000, 32, False), (32000, 4096, 32, False),
                                               (32000, 4096, 17, True)])
def test_noalloc_matches_the_oracle_and_the_allocating_entry_point_twice(lib, M, K, rows, out_bf16):
    from eagle_speculative_decoding_draft_gb300.engine import linear_bf16
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(M + K + rows)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for call in range(2):
        w = torch.from_numpy((rng.standard_normal((M, K)) / np.sqrt(K)).astype(np.float32)).to(
            torch.bfloat16).to(dev)
        x = torch.from_numpy(rng.standard_normal((rows, K)).astype(np.float32)).to(
            torch.bfloat16).to(dev)
        b = torch.from_numpy((rng.standard_normal(M) * 0.1).astype(np.float32)).to(
            torch.bfloat16).to(dev)
        ref = linear_bf16(w, x, b, out_bf16=out_bf16)
        got = _noalloc(lib, w, x, b, out_bf16)
        torch.cuda.synchronize()
        r = ref.double().cpu().numpy()
        g = got.double().cpu().numpy()
        if num_sms <= 160:
            assert np.array_equal(g, r), f"call {call}: not bit-identical to eagle_linear_bf16"
        wc, xf = w.cpu(), x.float().cpu().numpy()
        bf = b.double().cpu().numpy()
        absdot = np.abs(xf.astype(np.float64)) @ np.abs(wc.double().numpy()).T
        for i in range(rows):
            o = oracle.lm_head_row(wc, xf[i], True).astype(np.float64) + bf
            bound = 2 * gamma(K + 1) * (absdot[i] + np.abs(bf)) + 1e-30
            if out_bf16:
                bound = bound + 2.0 ** -8 * (np.abs(o) + bound)
            assert np.all(np.abs(g[i] - o) <= bound), f"call {call} row {i}: beyond the oracle's bound"
            assert np.all(np.abs(g[i] - r[i]) <= 2 * bound), f"call {call} row {i}"


def test_noalloc_refuses_oversize_requests(lib):
    P = ctypes.c_void_p
    assert lib.eagle_linear_noalloc_scratch_bytes() > 0
    # 33 rows, and 131073 output features, are beyond the fixed scratch
    assert lib.eagle_linear_bf16_noalloc(P(256), 64, P(256), 64, None, 128, 64, 33, P(256), 128, 0,
                                         None) == 1
    assert lib.eagle_linear_bf16_noalloc(P(256), 64, P(256), 64, None, 131073, 64, 8, P(256),
                                         131073, 0, None) == 1
