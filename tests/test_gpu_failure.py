"""Failure detection without a GPU fault: a device wait that nothing will satisfy gives up after
its limit, the kernel reports EAGLE_ERR_DEVICE_TIMEOUT through the status word and returns, and
the context stays usable (a GEMM launched afterwards is still correct and deterministic)."""
import ctypes
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    return torch.device("cuda", 0)


def test_bounded_wait_times_out_and_the_context_survives(dev):
    from eagle_speculative_decoding_draft_gb300 import _lib
    from eagle_speculative_decoding_draft_gb300.engine import linear_bf16
    lib = _lib.load()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for limit_ns in (1_000, 1_000_000, 20_000_000):
        t0 = time.perf_counter()
        rc = lib.eagle_test_bounded_wait(limit_ns, ctypes.c_void_p(status.data_ptr()), st)
        dt = time.perf_counter() - t0
        assert rc == 5, rc  # EAGLE_ERR_DEVICE_TIMEOUT
        assert dt >= limit_ns * 1e-9 * 0.5
        assert int(status.item()) == 0  # read and cleared
    # the context is intact: a GEMM afterwards matches a float64 reference
    rng = np.random.default_rng(0)
    W = torch.from_numpy((rng.standard_normal((300, 640)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    X = torch.from_numpy(rng.standard_normal((7, 640)).astype(np.float32)).to(torch.bfloat16)
    y = linear_bf16(W.to(dev), X.to(dev)).cpu().double()
    ref = X.double() @ W.double().T
    assert torch.allclose(y, ref, atol=1e-3, rtol=1e-3)


def test_bounded_wait_rejects_bad_arguments(dev):
    from eagle_speculative_decoding_draft_gb300 import _lib
    lib = _lib.load()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    P = ctypes.c_void_p
    assert lib.eagle_test_bounded_wait(0, P(status.data_ptr()), None) == 1
    assert lib.eagle_test_bounded_wait(10**11, P(status.data_ptr()), None) == 1
    assert lib.eagle_test_bounded_wait(1000, None, None) == 1
