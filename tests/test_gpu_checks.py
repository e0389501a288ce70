"""The small GPU parity cases on the checking build (-DEAGLE_CHECKS).

That build compiles in device-side checks of the kernels' own index invariants (a frontier's
candidates, a producing row, a gathered source row, a split-K slot, a tile ticket); a failed check
latches EAGLE_ERR_DEVICE_BOUNDS in the handle's status word, which every test reads.  This test
builds it and runs, in a child process that loads it (EAGLE_TREE_LIB), the component parity
tests (expand/build, verify, every way the streamed-weight GEMM splits its work), the small
end-to-end shapes, draft extend, static trees and the output guard words: all must pass with no
check failing."""
import os
import subprocess
import sys
from pathlib import Path

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parents[1]


def test_small_cases_pass_on_the_checking_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from eagle_speculative_decoding_draft_gb300 import build
    lib = build.build(checks=True)
    env = dict(os.environ, EAGLE_TREE_LIB=str(lib))
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
           "tests/test_gpu_canaries.py", "tests/test_gpu_extend.py", "tests/test_gpu_static.py",
           "tests/test_gpu_kernels.py::test_expand_and_build_are_bit_exact_on_oracle_inputs",
           "tests/test_gpu_kernels.py::test_verify_walk_and_greedy_are_bit_exact",
           "tests/test_gpu_kernels.py::test_linear_within_fp32_bound_of_oracle",
           "tests/test_gpu_parity.py::test_tiny_fp32_workload", "tests/test_gpu_parity.py::test_edge_shapes",
           "-k", "not 7b and not vicuna"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = (p.stdout + p.stderr)[-3000:]
    assert p.returncode == 0, tail
    assert " passed" in p.stdout, tail
