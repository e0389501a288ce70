"""The benchmark's host-side arithmetic, on the CPU: per-level GEMM figures, the static tree shape
rule, the clock summary, the GPU index under CUDA_VISIBLE_DEVICES, and the link between the
GEMM source and its recorded ncu traffic."""
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402


def test_per_level_means_and_fractions():
    plist = [
        {"level": 1, "kind": "fc", "ms": 0.020, "bytes": 60e6, "flops": 1e9},
        {"level": 1, "kind": "fc", "ms": 0.030, "bytes": 90e6, "flops": 2e9},
        {"level": 0, "kind": "lm_head", "ms": 0.050, "bytes": 250e6, "flops": 5e9},
    ]
    out = bench.per_level(plist, hbm=5000.0, tflops=1000.0)
    assert [(e["level"], e["kind"]) for e in out] == [(0, "lm_head"), (1, "fc")]
    fc = out[1]
    assert fc["launches"] == 2
    assert fc["us"] == pytest.approx(25.0)
    assert fc["GB/s"] == pytest.approx(150e6 / 50e-6 / 1e9)        # 3000 GB/s
    assert fc["hbm_frac"] == pytest.approx(0.6)
    assert fc["TFLOP/s"] == pytest.approx(3e9 / 50e-6 / 1e12)      # 60 TFLOP/s
    assert fc["tensor_frac"] == pytest.approx(0.06)
    assert out[0]["GB/s"] == pytest.approx(5000.0) and out[0]["hbm_frac"] == pytest.approx(1.0)


def test_static_shape_worked_example():
    # widths 4, 3, 2: the root takes 4; of depth 1, node 1 takes ceil(3/2) = 2 and node 2 the last
    # one; of depth 2, node 5 takes ceil(2/2) = 1 and node 6 the last one
    assert bench.static_widths(3, 4) == [4, 3, 2]
    assert bench.static_shape(3, 4) == [(0, 0), (0, 1), (0, 2), (0, 3), (1, 0), (1, 1), (2, 0), (5, 0), (6, 0)]


@pytest.mark.parametrize("depth,topk", [(6, 10), (5, 4), (5, 8), (1, 1), (4, 1), (32, 16)])
def test_static_shape_is_a_valid_tree(depth, topk):
    spec = bench.static_shape(depth, topk)
    widths = bench.static_widths(depth, topk)
    assert len(spec) == sum(widths)
    dep = [0]
    seen = set()
    for j, (p, r) in enumerate(spec, start=1):
        assert 0 <= p < j                      # parents first
        assert 0 <= r < 16 and (p, r) not in seen
        seen.add((p, r))
        dep.append(dep[p] + 1)
    assert [dep[1:].count(l + 1) for l in range(depth)] == widths
    assert all(b >= a for a, b in zip(dep, dep[1:]))   # depth never decreases


def test_clock_summary_parses_nvidia_smi_rows():
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 950.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c.lines = []
    assert c.summary()["samples"] == 0


def test_visible_gpu_index(monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.visible_gpu_index(0) == 3 and bench.visible_gpu_index(1) == 5
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.visible_gpu_index(2) == 2


def test_kernel_hash_ignores_comments_and_follows_code(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("int f(int x) {\n    return x + 1;\n}\n")
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ["k.cu"])
    h0 = bench.kernel_hash()
    src.write_text("// a note\nint f(int x) {  // why\n\n    /* more\n       words */\n    return x + 1;\n}\n")
    assert bench.kernel_hash() == h0
    src.write_text("int f(int x) {\n    return x + 2;\n}\n")
    assert bench.kernel_hash() != h0


def test_recorded_traffic_needs_the_current_hash(tmp_path, monkeypatch):
    import json
    src = tmp_path / "k.cu"
    src.write_text("int f() { return 1; }\n")
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ["k.cu"])
    prof = tmp_path / "t.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", prof)
    assert bench.recorded_traffic("w") is None                     # no record
    prof.write_text(json.dumps({"kernel_source_hash": bench.kernel_hash(),
                                "workloads": {"w": {"traffic_bytes_per_launch": 167.2e6}}}))
    assert bench.recorded_traffic("w") == pytest.approx(167.2e6)
    assert bench.recorded_traffic("other") is None                 # not captured for that one
    src.write_text("int f() { return 2; }\n")                     # the kernel changed since
    assert bench.recorded_traffic("w") is None


def test_step_floor_matches_the_survey_table():
    from eagle_speculative_decoding_draft_gb300 import synth
    # Vicuna-7B shape: 6 levels of 329.25 MB of weights, HBM-bound, about 291 us at 6779.4 GB/s
    f = bench.step_floor(synth.WORKLOADS[2], 6779.4, 1679.0)
    assert f["bytes"] == pytest.approx(1.976e9, rel=2e-3)
    assert f["us"] == pytest.approx(291.4, rel=3e-3)
    # Llama-3-8B vocabulary: 5 levels of 1117.8 MB; the 256-row levels sit near the ridge
    f5 = bench.step_floor(synth.WORKLOADS[5], 6779.4, 1679.0)
    assert f5["bytes"] == pytest.approx(5.589e9, rel=5e-3)
    assert 824.0 <= f5["us"] <= 900.0
    assert f5["verify_scan_bytes"] == 32 * 65 * 128256 * 2


def test_gemm_roofline_fractions():
    plist = [{"ms": 0.05, "bytes": 250e6, "flops": 1e9}, {"ms": 0.1, "bytes": 250e6, "flops": 150e12 * 1e-4}]
    r = bench.gemm_roofline(plist, hbm=5000.0, tflops=1000.0)
    assert r["achieved"] == pytest.approx(500e6 / 0.15e-3 / 1e9)
    # floors: 0.05 ms (bytes) and max(0.05, 0.015) ms: 0.1 ms of 0.15 ms measured
    assert r["frac_of_roofline_time"] == pytest.approx(0.1 / 0.15)
    assert bench.gemm_roofline([], 5000.0, 1000.0) is None
