#!/usr/bin/env python
"""Throughput of one EAGLE-2 dynamic draft-tree step on GB300.

A step is the whole hot path over one batch: d draft levels (gather, FC, LM head, log-softmax +
top-k, expand), the rerank + tree build, and greedy verification (target argmax + walk).  Every
run measures all five workloads; the headline (the JSON line's top-level figures) is the largest,
the Llama-3-8B vocabulary (h=4096, V=128256, batch 32, depth 5, k=8, m=64), and the other four
sit under "configs" with the same fields.  Inputs are seeded synthetic data; target logits are
the draft's own logits of every tree node plus N(0, sigma) noise, in bf16 for the bf16 workloads
(the dtype a bf16 target model emits; fp32-target figures are reported beside them).  Prints one
JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5] [--only]
                  [--impl eagle|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "draft-tree steps/sec (tree nodes/sec) at 1 GB300; % HBM or tensor roofline"
UNIT = "steps/s"
PEAKS_FILE = ROOT / "MEASURED_PEAKS.json"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
TRAFFIC_FILE = ROOT / "profiles" / "gemm_traffic.json"
KERNEL_SOURCES = ["eagle_speculative_decoding_draft_gb300/csrc/gemm.cu",
                  "eagle_speculative_decoding_draft_gb300/csrc/common.cuh"]
N_INPUT_SETS = 4
PROFILE_EVERY = 16
HEADLINE = 5            # the largest single-GPU workload: Llama-3-8B vocabulary
ORDER = [5, 1, 2, 3, 4]


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", type=int, default=HEADLINE,
                   help="the headline workload (1..5); the others follow under 'configs'")
    p.add_argument("--only", action="store_true", help="measure the headline workload alone")
    p.add_argument("--impl", choices=["eagle", "reference"], default="eagle")
    p.add_argument("--cpu-seconds", type=float, default=5.0,
                   help="wall-clock budget of the oracle's timed sample (all cores), per workload")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=100)
    p.add_argument("--side-figures", choices=["all", "headline", "none", "decoder"], default="all",
                   help="workloads that also time extend rounds, static trees, sampling and "
                        "greedy verification alone and the draft decoder layer (decoder: every "
                        "measured workload times the draft decoder layer alone)")
    p.add_argument("--decoder-requests", type=int, default=0,
                   help="run the draft decoder layer figure on the first N requests of the step's "
                        "tree (0: all of them); a smaller case for profiling its kernels")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Ranks:
    """The ranks of one run, from torchrun's environment (a single rank without it): a barrier,
    the max and the sum over ranks of a host number, and whole-job throughput.  Requests are
    independent, so every rank runs its own replica on its own inputs and nothing on the data
    path is exchanged; these reductions only combine the timings and counts."""

    def __init__(self, backend: str, device):
        self.world, self.rank, self.local = dist_env()
        self.device = device
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def _reduce(self, x: float, op_name: str) -> float:
        if self.dist is None:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=getattr(self.dist.ReduceOp, op_name))
        return float(t.item())

    def max(self, x: float) -> float:
        return self._reduce(x, "MAX")

    def sum(self, x: float) -> float:
        return self._reduce(x, "SUM")

    def throughput(self, units: float, seconds: float) -> float:
        """The units all ranks processed over the slowest rank's time."""
        return self.sum(units) / self.max(seconds)

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


def kernel_hash() -> str:
    """Hash of the GEMM's source code with comments and blank lines left out, so that the ncu
    counters recorded for it stay attached until the code itself changes."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        text = (ROOT / rel).read_text()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """dram read+write bytes per GEMM launch of `workload` from the committed ncu record
    (profiles/gemm_traffic.json), or None when there is none for it or the kernel source changed
    since that capture."""
    try:
        rec = json.loads(TRAFFIC_FILE.read_text())
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_hash") != kernel_hash():
        return None
    ent = rec.get("workloads", {}).get(workload)
    if not ent or "traffic_bytes_per_launch" not in ent:
        return None
    return float(ent["traffic_bytes_per_launch"])


def hbm_peak():
    try:
        return float(json.loads(PEAKS_FILE.read_text())["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Sustained dense bf16 TFLOP/s: the GEMM launches run inside a long loop of steps."""
    try:
        return float(json.loads(PEAKS_FILE.read_text())["bf16_tflops_sustained"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def static_widths(depth: int, topk: int):
    """Children per depth of the bench's static tree: topk at the root's depth, one fewer per
    level below, at least 1."""
    return [max(1, topk - l) for l in range(depth)]


def static_shape(depth: int, topk: int):
    """A static (EAGLE-1-style) tree for the bench: the nodes of each depth (its width) are shared
    out over the previous depth's nodes, best first: the i-th (0-based) gets about width / 2^(i+1)
    children (at least 1) until the width is used up, the last one the rest.  Returns (parent,
    rank) pairs."""
    spec = []
    prev = [0]  # nodes of the previous depth, best first
    for width in static_widths(depth, topk):
        cur = []
        budget = width
        for i, p in enumerate(prev):
            if budget <= 0:
                break
            last = i == len(prev) - 1
            kids = budget if last else min(budget, max(1, (width + (1 << (i + 1)) - 1) >> (i + 1)))
            for r in range(kids):
                spec.append((p, r))
                cur.append(len(spec))
            budget -= kids
        prev = cur
    return spec


def per_level(plist, hbm, tflops):
    """Mean duration, GB/s and TFLOP/s of the timed GEMM launches, by (level, kind)."""
    agg = {}
    for e in plist:
        a = agg.setdefault((e["level"], e["kind"]), [0, 0.0, 0.0, 0.0])
        a[0] += 1
        a[1] += e["ms"]
        a[2] += e["bytes"]
        a[3] += e["flops"]
    out = []
    for (lvl, kind), (c, ms, by, fl) in sorted(agg.items()):
        gbs = by / (ms * 1e-3) / 1e9
        tfs = fl / (ms * 1e-3) / 1e12
        out.append({"level": lvl, "kind": kind, "launches": c, "us": 1e3 * ms / c,
                    "GB/s": gbs, "hbm_frac": gbs / hbm, "TFLOP/s": tfs, "tensor_frac": tfs / tflops})
    return out


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def visible_gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
    return local_rank


# ----------------------------------------------------------------------------------------------
# The CPU oracle, timed on this host's cores (CPU-baseline leg and the reference arm)
# ----------------------------------------------------------------------------------------------

def oracle_sample(w, inp):
    """A bounded sample of the workload for the oracle: the first r requests (r = 1 unless the
    whole batch is small), with their target logits (oracle node logits + noise, untimed)."""
    import oracle

    r = w.batch if w.batch * w.num_nodes * w.hidden <= 4096 * 64 else 1
    idx = list(range(r))
    feat = inp.root_feat[idx].contiguous()
    tok = inp.root_tok[idx].contiguous()
    ref = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, feat, tok, w.depth, w.topk,
                            w.num_keep, w.is_bf16, rows=False, node_logits=True)
    rng = np.random.default_rng(4242)
    T = ref["node_z"] + rng.standard_normal(ref["node_z"].shape, dtype=np.float32) * np.float32(
        w.target_sigma)
    return r, feat, tok, T.astype(np.float32)


def time_oracle(w, inp, sample, budget_s, max_steps=None, warmup=0):
    """Runs the oracle's draft-tree step + greedy verify on the sample until the wall-clock budget
    (or max_steps) is used; returns (steps of the sample, seconds)."""
    import oracle

    r, feat, tok, T = sample

    def one():
        out = oracle.draft_tree(inp.w_fc, inp.b_fc, inp.w_lm, inp.emb, feat, tok, w.depth, w.topk,
                                w.num_keep, w.is_bf16, rows=False)
        oracle.verify_greedy(out["tree_tok"], out["tree_parent"], T, w.depth)

    for _ in range(warmup):
        one()
    n = 0
    t0 = time.perf_counter()
    while True:
        one()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps is not None and n >= max_steps):
            break
    return n, el


def cpu_baseline(w, inp, budget_s, one_thread=False):
    """The oracle on this host's cores (all of them, and on request also one thread) over a
    bounded sample of the workload; steps/s scaled to whole steps."""
    import oracle

    sample = oracle_sample(w, inp)
    r = sample[0]
    n, el = time_oracle(w, inp, sample, budget_s)
    value = n * r / w.batch / el
    out = {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"{n} oracle draft-tree steps (draft levels, rerank/build, greedy verify) of "
                     f"{r} of {w.batch} request(s), {el:.1f} s wall; value scaled to whole steps"}
    if one_thread:
        cores = oracle.num_threads()
        oracle.set_num_threads(1)
        try:
            n1, el1 = time_oracle(w, inp, sample, budget_s)
        finally:
            oracle.set_num_threads(cores)
        out["value_1_thread"] = n1 * r / w.batch / el1
        out["sample_1_thread"] = (f"{n1} steps of {r} of {w.batch} request(s) on one thread, "
                                  f"{el1:.1f} s wall")
    return out


def layer_dims(w):
    """(heads, kv_heads, head_dim, inter) of the target model's decoder layer that the draft layer
    copies, by workload shape; None for the fp32 toy (the layer is bf16 only)."""
    if not w.is_bf16:
        return None
    if w.hidden == 8192:
        return 64, 8, 128, 28672      # Llama-2-70B
    if w.vocab >= 128000:
        return 32, 8, 128, 14336      # Llama-3-8B
    return 32, 32, 128, 11008         # Llama-2-7B / Vicuna-7B


DECODER_PREFIX = 1024  # cached tokens per request in front of the tree


def decoder_layer_figure(w, dev, tree_out, rank, calls=200, requests=0):
    """The draft decoder layer over the step's tree: every node of every request, its mask and
    depth positions from the tree build, a DECODER_PREFIX-token KV cache per request.  Synthetic
    bf16 weights N(0, 1/sqrt(fan-in)), inputs and caches N(0, 1).  CUDA events over `calls` calls
    (weights and caches exceed L2, so every call reads them from HBM)."""
    import torch
    from eagle_speculative_decoding_draft_gb300.engine import DecoderLayer
    dims = layer_dims(w)
    if dims is None:
        return None
    H, Hk, D, I = dims
    h, B, n, P = w.hidden, w.batch, w.num_nodes, DECODER_PREFIX
    if 0 < requests < B:
        B = requests
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242 + rank)
    bf = lambda *shape, s=1.0: (torch.randn(*shape, generator=gen, device=dev) * s).to(torch.bfloat16)
    lay = DecoderLayer(bf((H + 2 * Hk) * D, h, s=h ** -0.5), bf(h, H * D, s=(H * D) ** -0.5),
                       (1 + 0.1 * torch.randn(h, generator=gen, device=dev)).to(torch.bfloat16),
                       bf(2 * I, h, s=h ** -0.5), bf(h, I, s=I ** -0.5), H, Hk)
    x = bf(B, n, h)
    kc, vc = bf(B, P, Hk, D), bf(B, P, Hk, D)
    pos = (tree_out["positions"][:B] + P).contiguous()
    mask = tree_out["mask"][:B].contiguous()
    out = torch.empty_like(x)
    for _ in range(5):
        lay(x, kc, vc, pos, mask, out=out, new_kv=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(calls):
        lay(x, kc, vc, pos, mask, out=out, new_kv=True)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / calls
    rows = B * n
    weight_bytes = 2 * h * ((H + 2 * Hk) * D + H * D + 3 * I)
    cache_bytes = 2 * 2 * B * P * Hk * D
    io_bytes = 2 * 2 * rows * h + 2 * 2 * rows * Hk * D + 4 * rows + 4 * rows * mask.shape[-1]
    total = weight_bytes + cache_bytes + io_bytes
    # projections: 2 flops per weight and row; attention: q.k and p.v over the cached keys and the
    # node's ancestors (at most depth + 1 tree keys) for every query head
    flops = 2.0 * rows * weight_bytes / 2 + 4.0 * rows * H * D * (P + w.depth + 1)
    return {"us_per_call": us, "achieved_gbs": total / (us * 1e-6) / 1e9,
            "flops_per_call": flops, "tflops": flops / (us * 1e-6) / 1e12,
            "algorithmic_bytes_per_call": total, "rows": rows, "prefix": P,
            "layer": {"heads": H, "kv_heads": Hk, "head_dim": D, "inter": I},
            "how": "eagle_decoder_layer over the step's tree (mask and positions from the build), "
                   f"new keys/values written; CUDA events, {calls} calls; bytes = weights + KV cache "
                   "+ layer input/output + new keys/values + positions/mask"}


def workload_config(w):
    mb = (2 * w.hidden * w.hidden + w.vocab * w.hidden) * (2 if w.is_bf16 else 4) / 1e6
    l2 = (f"inputs larger than L2: each level streams {mb:.0f} MB of weights (L2 is 129 MB); "
          "no flush") if mb > 129 else f"weights ({mb:.1f} MB) fit in L2: L2-resident timing"
    return {"workload": w.name, "hidden": w.hidden, "vocab": w.vocab, "batch": w.batch,
            "depth": w.depth, "topk": w.topk, "num_keep": w.num_keep,
            "tree_nodes_per_request": w.num_nodes, "global_batch": w.batch,
            "target_logits": "bf16" if w.is_bf16 else "f32",
            "parallelism": "replicas (one independent engine per GPU)", "l2": l2}


def step_floor(w, hbm_gbs, tflops):
    """The step's roofline floor in microseconds, as the survey's measurement table counts it:
    every level streams the FC and LM-head weights once (2h^2 + Vh elements) plus its gathered
    rows and top-k outputs; a level costs max(bytes / HBM, flops / tensor).  Also returned: the
    greedy verification's arg-max scan over the target logits (B (m+1) V elements)."""
    eb = 2 if w.is_bf16 else 4
    B, h, V, k, d = w.batch, w.hidden, w.vocab, w.topk, w.depth
    us = 0.0
    total_bytes = 0.0
    for l in range(d):
        R = B if l == 0 else B * k
        by = (2 * h * h + V * h) * eb + R * 2 * h * eb + R * (2 * k + 2) * 4
        fl = 2.0 * (2 * h * h + V * h) * R
        total_bytes += by
        us += max(by / (hbm_gbs * 1e3), fl / (tflops * 1e6))
    scan = B * w.num_nodes * V * (2 if w.is_bf16 else 4)
    return {"us": us, "bytes": total_bytes, "verify_scan_bytes": scan,
            "us_with_verify_scan": us + scan / (hbm_gbs * 1e3)}


def gemm_roofline(plist, hbm, tflops):
    """The streamed-weight GEMM's roofline over its timed launches: achieved GB/s against the HBM
    peak (the bound for every workload's launches taken together: their weight bytes over the HBM
    peak exceed their flops over the tensor peak), and the fraction of the per-launch roofline
    time, sum of max(bytes / HBM, flops / tensor) over the measured time."""
    ms = sum(e["ms"] for e in plist)
    by = sum(e["bytes"] for e in plist)
    fl = sum(e["flops"] for e in plist)
    if ms <= 0:
        return None
    floor_ms = sum(max(e["bytes"] / (hbm * 1e6), e["flops"] / (tflops * 1e9)) for e in plist)
    achieved = by / (ms * 1e-3) / 1e9
    return {"achieved": achieved, "frac": achieved / hbm, "ms": ms, "bytes": by, "flops": fl,
            "tflops_achieved": fl / (ms * 1e-3) / 1e12, "tensor_frac": fl / (ms * 1e-3) / 1e12 / tflops,
            "frac_of_roofline_time": floor_ms / ms, "hbm_bound_ms": by / (hbm * 1e6),
            "tensor_bound_ms": fl / (tflops * 1e9)}


def run_reference(args, w):
    """The reference arm: the oracle, as it stands, on this host's cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from eagle_speculative_decoding_draft_gb300 import synth

    inp = synth.make_inputs(w)
    sample = oracle_sample(w, inp)
    r = sample[0]
    budget = 150.0
    n, el = time_oracle(w, inp, sample, budget, max_steps=max(1, args.steps),
                        warmup=min(args.warmup, 1))
    value = n * r / w.batch / el
    cb = {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
          "sample": f"{n} oracle steps of {r} of {w.batch} request(s) in {el:.1f} s (at most "
                    f"{budget:.0f} s), value scaled to whole steps"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": n, "warmup": min(args.warmup, 1),
            "ms_per_step": 1e3 / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.is_bf16 else "f32", "data": "synthetic (seeded)",
            "config": workload_config(w), "tree_nodes_per_s": value * w.batch * w.num_nodes,
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------
# The GPU engine
# ----------------------------------------------------------------------------------------------

def timed(fn, calls):
    """Milliseconds per call of fn(i), CUDA events on the current stream around `calls` calls."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for i in range(calls):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / calls


def e2e_figure(eng, w, sets_host, steps, ranks):
    """Steps/s through eagle_tree_step_host: the step's inputs and target logits copied from
    pinned host memory and its results copied back, stream synchronised, every step."""
    import torch
    B, n, d, W = w.batch, w.num_nodes, w.depth, eng.mask_words
    staging = torch.empty(sets_host[0][2].shape, dtype=sets_host[0][2].dtype, device=eng.device)
    i32 = dict(dtype=torch.int32, pin_memory=True)
    hout = {"tokens": torch.empty(B, n, **i32), "parents": torch.empty(B, n, **i32),
            "positions": torch.empty(B, n, **i32), "mask": torch.empty(B, n, W, **i32),
            "accept_len": torch.empty(B, **i32), "accept_tokens": torch.empty(B, d + 1, **i32)}
    for i in range(3):
        f, t, T = sets_host[i % len(sets_host)]
        eng.step_host(f, t, T, staging, hout)
    ranks.barrier()
    t0 = time.perf_counter()
    for i in range(steps):
        f, t, T = sets_host[i % len(sets_host)]
        eng.step_host(f, t, T, staging, hout)
    value = ranks.throughput(steps, time.perf_counter() - t0)
    ranks.barrier()
    f, t, T = sets_host[0]
    h2d = f.numel() * f.element_size() + t.numel() * 4 + T.numel() * T.element_size()
    d2h = 4 * (3 * B * n + B * n * W + B + B * (d + 1))
    del staging
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "target_logits": "bf16" if T.dtype == torch.bfloat16 else "f32", "steps": steps,
            "graphed": eng.step_graphed() == 1,
            "how": "eagle_tree_step_host per step: pinned host inputs and target logits copied in, "
                   "tree and verify results copied out, stream synchronised"}


def decoder_only_figure(eng, w, sets, tree_out, ver_out, dev, rank, requests=0):
    """The draft decoder layer figure alone (over the tree of input set 0)."""
    feat0, tok0, T0 = sets[0][0], sets[0][1], sets[0][2]
    eng.step(feat0, tok0, T0, tree_out=tree_out, verify_out=ver_out)
    dec = decoder_layer_figure(w, dev, tree_out, rank, requests=requests)
    if dec is not None:
        peak, _ = hbm_peak()
        tp, _ = tensor_peak()
        dec["frac_of_hbm"] = dec["achieved_gbs"] / peak
        dec["frac_of_bf16_sustained"] = dec["tflops"] / tp
    return dec


def side_figures(eng, w, inp, sets, tree_out, ver_out, dev, rank, K, decoder_requests=0):
    """Figures beside the step: extend rounds, an EAGLE-1 static tree, sampling and greedy
    verification alone, and the draft decoder layer over the step's tree."""
    import torch
    from eagle_speculative_decoding_draft_gb300.engine import EagleTree, verify_sample
    B, h, V, n, d = w.batch, w.hidden, w.vocab, w.num_nodes, w.depth
    fdt = torch.bfloat16 if w.is_bf16 else torch.float32
    g = lambda t: t.to(dev).contiguous()
    out = {}
    peak, _ = hbm_peak()

    # sampling verification (recursive rejection sampling) on the tree of input set 0: q = the
    # draft's logits of every node, p = the target logits, temperature 1, fresh uniforms per call
    feat0, tok0, T0 = sets[0][0], sets[0][1], sets[0][2]
    eng.step(feat0, tok0, T0, tree_out=tree_out, verify_out=ver_out)
    Zn = eng.node_logits(feat0).contiguous()
    T0c = T0.float().contiguous()
    scratch = torch.empty(B, V, dtype=torch.float32, device=dev)
    ugen = torch.Generator(device=dev)
    ugen.manual_seed(77 + rank)
    S_CALLS = 50
    us = [(torch.rand(B, n, generator=ugen, device=dev), torch.rand(B, generator=ugen, device=dev))
          for _ in range(S_CALLS)]
    sacc = []

    def samp(i):
        o = verify_sample(tree_out["tokens"], tree_out["parents"], T0c, Zn, d, 1.0, us[i][0],
                          us[i][1], scratch=scratch)
        sacc.append(o["accept_len"])

    for i in range(3):
        samp(i)
    sacc.clear()
    sample_ms = timed(samp, S_CALLS)
    out["sampling_verify"] = {"us_per_call": sample_ms * 1e3,
                              "mean_accept_len": float(torch.stack(sacc).float().mean().item()),
                              "temperature": 1.0, "mode": "recursive rejection sampling",
                              "how": "eagle_verify_sample on the step's tree; q = draft logits of "
                                     "every node, p = the synthetic target (fp32); CUDA events, "
                                     f"{S_CALLS} calls"}
    del Zn, T0c, scratch, us

    # greedy verification alone, cycling over the input sets' target logits
    G_CALLS = 50
    gv = lambda i: eng.verify_greedy(tree_out["tokens"], tree_out["parents"], sets[i % N_INPUT_SETS][2],
                                     None, ver_out)
    for i in range(3):
        gv(i)
    greedy_us = timed(gv, G_CALLS) * 1e3
    greedy_bytes = float(T0.numel() * T0.element_size())
    out["greedy_verify"] = {"us_per_call": greedy_us, "target_logit_bytes": greedy_bytes,
                            "target_logits": "bf16" if T0.dtype == torch.bfloat16 else "f32",
                            "achieved_gbs": greedy_bytes / (greedy_us * 1e-6) / 1e9,
                            "frac_of_hbm": greedy_bytes / (greedy_us * 1e-6) / 1e9 / peak,
                            "target_logits_in_l2": N_INPUT_SETS * greedy_bytes <= 96e6,
                            "how": "eagle_verify_greedy (arg-max over the B x (m+1) x V target logits, "
                                   "then the walk) on the step's tree, alone; CUDA events, "
                                   f"{G_CALLS} calls over {N_INPUT_SETS} target sets; bytes = the "
                                   "target logits read (a roofline only when they exceed L2)"}

    # the multi-round loop with draft extend: each round starts from the previous verify through
    # eagle_draft_extend, then levels 1..d-1, the rerank/build and the greedy verify
    fgen = torch.Generator(device=dev)
    fgen.manual_seed(99 + rank)
    Fn = [torch.randn(B, n, h, generator=fgen, device=dev).to(fdt) for _ in range(2)]
    eng.step(feat0, tok0, T0, tree_out=tree_out, verify_out=ver_out)

    def one_round(i):
        eng.extend(Fn[i % 2], ver_out["accept_len"], ver_out["accept_nodes"], ver_out["accept_tokens"])
        for lvl in range(1, d):
            eng.draft_level(lvl)
        eng.rerank_build_tree(out=tree_out)
        eng.verify_greedy(tree_out["tokens"], tree_out["parents"], sets[i % N_INPUT_SETS][2], out=ver_out)

    for i in range(5):
        one_round(i)
    ROUNDS = max(50, K // 4)
    round_ms = timed(one_round, ROUNDS)
    eng.status()
    out["round_with_extend"] = {"value": 1e3 / round_ms, "unit": "rounds/s", "ms_per_round": round_ms,
                                "rounds": ROUNDS,
                                "how": "eagle_draft_extend from the previous verify (FC over every "
                                       "verified position + the next tree's level 0), levels 1..d-1, "
                                       "rerank/build, greedy verify; CUDA events, eager launches"}
    del Fn

    # an EAGLE-1 static tree on the same weights
    spec = static_shape(d, w.topk)
    st_eng = EagleTree(*eng._keep, B, d, 1, len(spec), static_spec=spec)
    st_n = len(spec) + 1
    st_T = [torch.randn(B, st_n, V, generator=fgen, device=dev).to(sets[0][2].dtype) for _ in range(2)]
    st_tree, st_ver = st_eng.new_tree_outputs(), st_eng.new_verify_outputs()

    def static_step(i):
        f_i, t_i = sets[i % N_INPUT_SETS][0], sets[i % N_INPUT_SETS][1]
        st_eng.step(f_i, t_i, st_T[i % 2], tree_out=st_tree, verify_out=st_ver)

    for i in range(5):
        static_step(i)
    static_ms = timed(static_step, max(50, K // 4))
    st_eng.status()
    st_eng.close()
    del st_T
    out["static_tree"] = {"value": 1e3 / static_ms, "unit": "steps/s", "ms_per_step": static_ms,
                          "drafted_nodes": len(spec), "depth": d, "shape": "widths " + str(static_widths(d, w.topk)),
                          "how": "eagle_tree_init_static handle on the same weights: levels, build, greedy "
                                 "verify against N(0,1) target logits; CUDA events, eager launches"}

    # the draft decoder layer over the step's tree
    eng.step(feat0, tok0, T0, tree_out=tree_out, verify_out=ver_out)
    dec = decoder_layer_figure(w, dev, tree_out, rank, requests=decoder_requests)
    if dec is not None:
        dec["frac_of_hbm"] = dec["achieved_gbs"] / peak
        tp, _ = tensor_peak()
        dec["frac_of_bf16_sustained"] = dec["tflops"] / tp
    out["draft_decoder_layer"] = dec
    return out


def measure(args, w, dev, ranks, rank, local, headline):
    """Every figure of one workload; returns its entry of the JSON line."""
    import torch

    from eagle_speculative_decoding_draft_gb300 import synth
    from eagle_speculative_decoding_draft_gb300.engine import EagleTree

    inp = synth.make_inputs(w)
    g = lambda t: t.to(dev).contiguous()
    w_fc, w_lm, emb = g(inp.w_fc), g(inp.w_lm), g(inp.emb)
    b_fc = g(inp.b_fc) if w.bias else None
    eng = EagleTree(w_fc, b_fc, w_lm, emb, w.batch, w.depth, w.topk, w.num_keep)
    B, h, V, n, d = w.batch, w.hidden, w.vocab, w.num_nodes, w.depth
    fdt = torch.bfloat16 if w.is_bf16 else torch.float32
    tdt = torch.bfloat16 if w.is_bf16 else torch.float32  # target logits as the target model emits them

    # a few distinct input batches, each with its synthetic target (draft logits + noise)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    sets, sets32 = [], []
    for i in range(N_INPUT_SETS):
        if i == 0:
            feat, tok = inp.root_feat, inp.root_tok
        else:
            rng = np.random.default_rng(5000 + 17 * i + rank)
            feat = torch.from_numpy(rng.standard_normal((B, h), dtype=np.float32)).to(fdt)
            tok = torch.from_numpy(rng.integers(0, V, size=B).astype(np.int32))
        feat, tok = g(feat), g(tok)
        eng.draft(feat, tok)
        T = eng.node_logits(feat)
        T.add_(torch.randn(T.shape, generator=gen, device=dev), alpha=w.target_sigma)
        sets.append((feat, tok, T.to(tdt) if tdt != torch.float32 else T))
        if tdt != torch.float32:
            sets32.append((feat, tok, T))
        else:
            sets32.append(sets[-1])
    tree_out, ver_out = eng.new_tree_outputs(), eng.new_verify_outputs()

    def step(i, s=sets):
        feat, tok, T = s[i % N_INPUT_SETS]
        eng.step(feat, tok, T, tree_out=tree_out, verify_out=ver_out)

    for i in range(max(args.warmup, 0)):
        step(i)
    eng.profile(64)
    step(0)
    gemm_per_step, _, _ = eng.profile_read()
    torch.cuda.synchronize()
    eng.status()

    # ---------------- eager launches, GEMM launches of 1 step in 16 bracketed by events ----------
    K = args.steps
    sampled = [i for i in range(K) if i % PROFILE_EVERY == 0]
    eng.profile(len(sampled) * gemm_per_step)
    l0 = eng.launch_count()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for i in range(K):
        eng.profile_enable(i % PROFILE_EVERY == 0)
        step(i)
    end.record()
    torch.cuda.synchronize()
    eng.profile_enable(True)
    eager_ms = start.elapsed_time(end)
    launches_per_step = (eng.launch_count() - l0) / K
    plist = eng.profile_list(len(sampled) * gemm_per_step)
    eng.profile(0)
    eng.status()

    # ---------------- CUDA graph: one captured step per input set, replayed ----------------
    cap = torch.cuda.Stream(device=dev)
    graphs, graphs32 = [], []
    try:
        with torch.cuda.stream(cap):
            for i in range(N_INPUT_SETS):
                step(i)  # warm the capture stream
        torch.cuda.synchronize()
        for lst, s in ((graphs, sets), (graphs32, sets32 if tdt != torch.float32 else None)):
            if s is None:
                continue
            for i in range(N_INPUT_SETS):
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=cap):
                    step(i, s)
                lst.append(gr)
        torch.cuda.synchronize()
        eng.status()
    except Exception as exc:  # a failed capture leaves the eager figure as the value
        graphs, graphs32 = [], []
        graph_error = repr(exc)[:200]
    else:
        graph_error = None
    for i in range(2 * N_INPUT_SETS):
        if graphs:
            graphs[i % N_INPUT_SETS].replay()
    torch.cuda.synchronize()

    with ClockSampler(visible_gpu_index(local)) as clocks:
        ranks.barrier()
        torch.cuda.synchronize()
        start.record()
        for i in range(K):
            if graphs:
                graphs[i % N_INPUT_SETS].replay()
            else:
                step(i)
        end.record()
        torch.cuda.synchronize()
        ranks.barrier()
    ms = start.elapsed_time(end)
    eng.status()
    value = ranks.throughput(K, ms / 1e3)
    ms_max = ranks.max(ms)
    value32 = None
    if graphs32:
        for i in range(N_INPUT_SETS):
            graphs32[i].replay()
        ms32 = timed(lambda i: graphs32[i % N_INPUT_SETS].replay(), K)
        value32 = ranks.throughput(K, ms32 * K / 1e3)
        eng.status()
    del graphs, graphs32

    accept = []
    for i in range(N_INPUT_SETS):
        step(i)
        accept.append(ver_out["accept_len"].float().mean().item())
    torch.cuda.synchronize()

    # ---------------- end to end through eagle_tree_step_host ----------------
    pin = lambda t: t.cpu().pin_memory()
    E = max(1, args.e2e_steps)
    e2e = e2e_figure(eng, w, [(pin(f), pin(t), pin(T)) for f, t, T in sets], E, ranks)
    e2e32 = None
    if tdt != torch.float32:
        e2e32 = e2e_figure(eng, w, [(pin(f), pin(t), pin(T)) for f, t, T in sets32[:2]],
                           max(1, E // 2), ranks)

    peak, peak_kind = hbm_peak()
    tpeak, tpeak_kind = tensor_peak()
    floor = step_floor(w, peak, tpeak)
    gr = gemm_roofline(plist, peak, tpeak)
    entry = {
        "value": value, "unit": UNIT, "ms_per_step": ms_max / K, "steps": K,
        "mode": ("CUDA graph replay (one captured step per input set), CUDA events on the replay "
                 "stream" if graph_error is None else f"eager launches (graph capture failed: {graph_error})"),
        "value_eager": ranks.throughput(K, eager_ms / 1e3),
        "value_fp32_target": value32,
        "tree_nodes_per_s": value * B * n,
        "mean_accept_len": float(np.mean(accept)),
        "config": workload_config(w),
        "step_floor_us": floor["us"], "step_floor_bytes": floor["bytes"],
        "step_frac_of_floor": floor["us"] / (1e3 * ms_max / K),
        "step_floor_us_with_verify_scan": floor["us_with_verify_scan"],
        "roofline": None if gr is None else {
            "bound": "hbm", "kernel": "linear_bf16_tc_kernel (FC and LM head)",
            "achieved": gr["achieved"], "peak": peak, "unit": "GB/s", "frac": gr["frac"],
            "peak_source": f"{peak_kind} hbm_gbs (of {peak_kind})",
            "traffic": recorded_traffic(w.name),
            "algorithmic_bytes_per_launch": gr["bytes"] / max(len(plist), 1),
            "launches_timed": len(plist), "ms_per_launch": gr["ms"] / max(len(plist), 1),
            "tflops_achieved": gr["tflops_achieved"], "tensor_frac": gr["tensor_frac"],
            "frac_of_roofline_time": gr["frac_of_roofline_time"],
            "timed_steps": f"GEMM launches of 1 eager step in {PROFILE_EVERY} (events stop those "
                           "launches overlapping their predecessor)",
            "gemm_ms_per_step_standalone": gr["ms"] / max(len(sampled), 1),
            "per_level": per_level(plist, peak, tpeak),
            "tensor_peak": tpeak, "tensor_peak_source": f"{tpeak_kind} bf16_tflops_sustained"},
        "clocks": clocks.summary(),
        "e2e": e2e, "e2e_fp32_target": e2e32,
        "gpu_launches_per_step": launches_per_step,
        "gpu_launches": int(ranks.sum(round(launches_per_step * K))),
    }
    if args.side_figures == "all" or (args.side_figures == "headline" and headline):
        entry.update(side_figures(eng, w, inp, sets, tree_out, ver_out, dev, rank, K,
                                  args.decoder_requests))
    elif args.side_figures == "decoder":
        entry["draft_decoder_layer"] = decoder_only_figure(eng, w, sets, tree_out, ver_out, dev, rank,
                                                           args.decoder_requests)
    eng.close()
    if rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        entry["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_seconds, one_thread=headline)
    del eng, sets, sets32, w_fc, w_lm, emb, b_fc, tree_out, ver_out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def run_eagle(args, order):
    import torch

    from eagle_speculative_decoding_draft_gb300 import synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks("nccl", dev)
    entries = []
    for num in order:
        entries.append((num, measure(args, synth.WORKLOADS[num], dev, ranks, rank, local,
                                     headline=num == order[0])))
    num0, top = entries[0]
    w0 = synth.WORKLOADS[num0]
    line = {
        "metric": METRIC, "value": top["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": top["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w0.is_bf16 else "f32",
        "data": "synthetic (seeded); target logits = the draft's logits of every tree node + "
                f"N(0, sigma), bf16 for the bf16 workloads",
        "config": top["config"],
        "roofline": top["roofline"], "clocks": top["clocks"], "e2e": top["e2e"],
        "gpu_launches": top["gpu_launches"],
        "gpu_launches_all_workloads": int(sum(e["gpu_launches"] for _, e in entries)),
    }
    if "cpu_baseline" in top:
        line["cpu_baseline"] = top["cpu_baseline"]
    for key, val in top.items():
        if key not in line and key not in ("config", "unit", "steps"):
            line[key] = val
    line["configs"] = {synth.WORKLOADS[num].name: e for num, e in entries[1:]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    ranks.close()


def main():
    args = parse_args()
    from eagle_speculative_decoding_draft_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        order = [args.workload] if args.only else [args.workload] + [n for n in ORDER if n != args.workload]
        run_eagle(args, order)


if __name__ == "__main__":
    main()
