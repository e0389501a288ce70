#!/usr/bin/env python
"""Throughput of one EAGLE-2 dynamic draft-tree step on GB300.

A step is the whole hot path over one batch: d draft levels (gather, FC, LM head, log-softmax +
top-k, expand), the rerank + tree build, and greedy verification (target argmax + walk).  The
default workload is the Vicuna-7B shape (h=4096, V=32000, batch 1, depth 6, k=10, m=60).
Inputs are seeded synthetic data; target logits are the draft's own logits of every tree node
plus N(0, sigma) noise.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5] [--impl eagle|reference]
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
TRAFFIC_FILE = ROOT / "profiles" / "linear_bf16_tc_vicuna7b.md"
KERNEL_SOURCES = ["eagle_speculative_decoding_draft_gb300/csrc/gemm.cu",
                  "eagle_speculative_decoding_draft_gb300/csrc/common.cuh"]
N_INPUT_SETS = 4
PROFILE_EVERY = 16


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--workload", type=int, default=2)
    p.add_argument("--impl", choices=["eagle", "reference"], default="eagle")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="wall-clock budget of the oracle's timed sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=300)
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


def recorded_traffic():
    """dram read+write bytes per GEMM launch from the committed ncu summary, or None when the
    kernel source changed since that capture."""
    if not TRAFFIC_FILE.exists():
        return None
    text = TRAFFIC_FILE.read_text()
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_val = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_val or m_hash.group(1) != kernel_hash():
        return None
    return float(m_val.group(1))


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


def cpu_baseline(w, inp, budget_s):
    import oracle

    sample = oracle_sample(w, inp)
    r = sample[0]
    n, el = time_oracle(w, inp, sample, budget_s)
    value = n * r / w.batch / el
    return {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} oracle draft-tree steps (draft levels, rerank/build, greedy verify) of "
                      f"{r} of {w.batch} request(s), {el:.1f} s wall; value scaled to whole steps"}


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


def decoder_layer_figure(w, dev, tree_out, rank, calls=200):
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
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242 + rank)
    bf = lambda *shape, s=1.0: (torch.randn(*shape, generator=gen, device=dev) * s).to(torch.bfloat16)
    lay = DecoderLayer(bf((H + 2 * Hk) * D, h, s=h ** -0.5), bf(h, H * D, s=(H * D) ** -0.5),
                       (1 + 0.1 * torch.randn(h, generator=gen, device=dev)).to(torch.bfloat16),
                       bf(2 * I, h, s=h ** -0.5), bf(h, I, s=I ** -0.5), H, Hk)
    x = bf(B, n, h)
    kc, vc = bf(B, P, Hk, D), bf(B, P, Hk, D)
    pos = (tree_out["positions"] + P).contiguous()
    mask = tree_out["mask"].contiguous()
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
    return {"us_per_call": us, "achieved_gbs": total / (us * 1e-6) / 1e9,
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
            "parallelism": "replicas (one independent engine per GPU)", "l2": l2}


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

def run_eagle(args, w):
    import torch

    from eagle_speculative_decoding_draft_gb300 import synth
    from eagle_speculative_decoding_draft_gb300.engine import EagleTree

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks("nccl", dev)
    barrier = ranks.barrier

    inp = synth.make_inputs(w)
    g = lambda t: t.to(dev).contiguous()
    eng = EagleTree(g(inp.w_fc), g(inp.b_fc) if w.bias else None, g(inp.w_lm), g(inp.emb),
                    w.batch, w.depth, w.topk, w.num_keep)
    B, h, V, n, d = w.batch, w.hidden, w.vocab, w.num_nodes, w.depth
    fdt = torch.bfloat16 if w.is_bf16 else torch.float32

    # a few distinct input batches, each with its synthetic target (draft logits + noise)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    sets = []
    for i in range(N_INPUT_SETS):
        if i == 0:
            feat, tok = inp.root_feat, inp.root_tok
        else:
            rng = np.random.default_rng(5000 + 17 * i + rank)
            feat = torch.from_numpy(rng.standard_normal((B, h), dtype=np.float32)).to(fdt)
            tok = torch.from_numpy(rng.integers(0, V, size=B).astype(np.int32))
        feat, tok = g(feat), g(tok)
        eng.draft(feat, tok)
        nz = eng.node_logits(feat)
        T = nz + w.target_sigma * torch.randn(nz.shape, generator=gen, device=dev)
        sets.append((feat, tok, T))
    tree_out, ver_out = eng.new_tree_outputs(), eng.new_verify_outputs()

    def step(i):
        feat, tok, T = sets[i % N_INPUT_SETS]
        eng.step(feat, tok, T, tree_out=tree_out, verify_out=ver_out)

    for i in range(max(args.warmup, 0)):
        step(i)
    eng.profile(64)
    step(0)
    gemm_per_step, _, _ = eng.profile_read()
    torch.cuda.synchronize()
    eng.status()

    # ---------------- timed region: K steps, device time ----------------
    # The GEMM launches of one step in PROFILE_EVERY are bracketed by CUDA events (the kernel's
    # own duration); events keep a launch from overlapping its predecessor, so the other steps
    # run without them.
    K = args.steps
    sampled = [i for i in range(K) if i % PROFILE_EVERY == 0]
    eng.profile(len(sampled) * gemm_per_step)
    l0 = eng.launch_count()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(visible_gpu_index(local)) as clocks:
        barrier()
        torch.cuda.synchronize()
        start.record()
        for i in range(K):
            eng.profile_enable(i % PROFILE_EVERY == 0)
            step(i)
        end.record()
        torch.cuda.synchronize()
        barrier()
    eng.profile_enable(True)
    ms = start.elapsed_time(end)
    launches = eng.launch_count() - l0
    plist = eng.profile_list(len(sampled) * gemm_per_step)
    n_prof = len(plist)
    gemm_ms = sum(e["ms"] for e in plist)
    gemm_bytes = sum(e["bytes"] for e in plist)
    eng.profile(0)
    eng.status()
    ms_max = ranks.max(ms)
    value = ranks.throughput(K, ms / 1e3)

    accept = []
    for i in range(N_INPUT_SETS):
        step(i)
        accept.append(ver_out["accept_len"].float().mean().item())
    torch.cuda.synchronize()

    # ---------------- end to end: host buffers through eagle_tree_step_host ----------------
    pin = lambda t: t.cpu().pin_memory()
    hsets = [(pin(f), pin(t), pin(T)) for f, t, T in sets]
    staging = torch.empty_like(sets[0][2])
    W = eng.mask_words
    i32 = dict(dtype=torch.int32, pin_memory=True)
    hout = {"tokens": torch.empty(B, n, **i32), "parents": torch.empty(B, n, **i32),
            "positions": torch.empty(B, n, **i32), "mask": torch.empty(B, n, W, **i32),
            "accept_len": torch.empty(B, **i32), "accept_tokens": torch.empty(B, d + 1, **i32)}
    for i in range(3):
        f, t, T = hsets[i % N_INPUT_SETS]
        eng.step_host(f, t, T, staging, hout)
    E = max(1, args.e2e_steps)
    barrier()
    t0 = time.perf_counter()
    for i in range(E):
        f, t, T = hsets[i % N_INPUT_SETS]
        eng.step_host(f, t, T, staging, hout)
    e2e_value = ranks.throughput(E, time.perf_counter() - t0)
    barrier()
    f, t, T = hsets[0]
    h2d = f.numel() * f.element_size() + t.numel() * 4 + T.numel() * T.element_size()
    d2h = 4 * (3 * B * n + B * n * W + B + B * (d + 1))

    # ---------------- sampling verification (recursive rejection sampling) ----------------
    # On the tree of input set 0: q = the draft's logits of every node, p = the target logits,
    # temperature 1, fresh uniforms per call.  Timed alone with CUDA events.
    from eagle_speculative_decoding_draft_gb300.engine import verify_sample
    feat0, tok0, T0 = sets[0]
    eng.step(feat0, tok0, T0, tree_out=tree_out, verify_out=ver_out)
    Zn = eng.node_logits(feat0).contiguous()
    T0c = T0.float().contiguous()
    scratch = torch.empty(B, w.vocab, dtype=torch.float32, device=dev)
    ugen = torch.Generator(device=dev)
    ugen.manual_seed(77 + rank)
    S_CALLS = 50
    us = [(torch.rand(B, n, generator=ugen, device=dev), torch.rand(B, generator=ugen, device=dev))
          for _ in range(S_CALLS)]
    sacc = []
    for i in range(3):
        verify_sample(tree_out["tokens"], tree_out["parents"], T0c, Zn, d, 1.0, us[i][0], us[i][1],
                      scratch=scratch)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for i in range(S_CALLS):
        o = verify_sample(tree_out["tokens"], tree_out["parents"], T0c, Zn, d, 1.0, us[i][0], us[i][1],
                          scratch=scratch)
        sacc.append(o["accept_len"])
    s1.record()
    torch.cuda.synchronize()
    sample_us = s0.elapsed_time(s1) * 1e3 / S_CALLS
    sample_accept = float(torch.stack(sacc).float().mean().item())

    # ---------------- greedy verification alone ----------------
    # The arg-max over every tree node's target logits and the walk, on the tree of input set 0,
    # cycling over the input sets' target logits (at the Llama-3-8B vocabulary they are 1.07 GB
    # each, far beyond L2; the smaller shapes' 4 sets stay in L2).  CUDA events, G_CALLS calls.
    G_CALLS = 50
    for i in range(3):
        eng.verify_greedy(tree_out["tokens"], tree_out["parents"], sets[i % N_INPUT_SETS][2], None, ver_out)
    torch.cuda.synchronize()
    s0.record()
    for i in range(G_CALLS):
        eng.verify_greedy(tree_out["tokens"], tree_out["parents"], sets[i % N_INPUT_SETS][2], None, ver_out)
    s1.record()
    torch.cuda.synchronize()
    greedy_us = s0.elapsed_time(s1) * 1e3 / G_CALLS
    greedy_bytes = float(T0.numel() * T0.element_size())
    in_l2 = N_INPUT_SETS * greedy_bytes <= 96e6

    # ---------------- the multi-round loop with draft extend ----------------
    # Steady state of decoding: each round starts from the previous verify through
    # eagle_draft_extend (the FC over every verified position, then level 0 of the next tree),
    # then levels 1..d-1, the rerank/build and the greedy verify.  Target features of the tree
    # nodes are synthetic N(0, 1); the target logits cycle over the input sets.
    fgen = torch.Generator(device=dev)
    fgen.manual_seed(99 + rank)
    Fn = [torch.randn(B, n, h, generator=fgen, device=dev).to(fdt) for _ in range(N_INPUT_SETS)]
    eng.step(feat0, tok0, T0, tree_out=tree_out, verify_out=ver_out)

    def one_round(i):
        _, _, Ti = sets[i % N_INPUT_SETS]
        eng.extend(Fn[i % N_INPUT_SETS], ver_out["accept_len"], ver_out["accept_nodes"],
                   ver_out["accept_tokens"])
        for lvl in range(1, d):
            eng.draft_level(lvl)
        eng.rerank_build_tree(out=tree_out)
        eng.verify_greedy(tree_out["tokens"], tree_out["parents"], Ti, out=ver_out)

    for i in range(10):
        one_round(i)
    ROUNDS = max(100, K // 4)
    torch.cuda.synchronize()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record()
    for i in range(ROUNDS):
        one_round(i)
    r1.record()
    torch.cuda.synchronize()
    round_ms = r0.elapsed_time(r1) / ROUNDS
    eng.status()

    # ---------------- an EAGLE-1 static tree on the same weights ----------------
    spec = static_shape(d, w.topk)
    st_eng = EagleTree(g(inp.w_fc), g(inp.b_fc) if w.bias else None, g(inp.w_lm), g(inp.emb), B,
                       d, 1, len(spec), static_spec=spec)
    st_n = len(spec) + 1
    st_T = [torch.randn(B, st_n, V, generator=fgen, device=dev) for _ in range(2)]
    st_tree, st_ver = st_eng.new_tree_outputs(), st_eng.new_verify_outputs()

    def static_step(i):
        feat_i, tok_i, _ = sets[i % N_INPUT_SETS]
        st_eng.step(feat_i, tok_i, st_T[i % 2], tree_out=st_tree, verify_out=st_ver)

    for i in range(10):
        static_step(i)
    torch.cuda.synchronize()
    s_0, s_1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    S_STEPS = max(100, K // 4)
    s_0.record()
    for i in range(S_STEPS):
        static_step(i)
    s_1.record()
    torch.cuda.synchronize()
    static_ms = s_0.elapsed_time(s_1) / S_STEPS
    st_eng.status()
    st_eng.close()

    # ---------------- the draft decoder layer over the step's tree ----------------
    eng.step(feat0, tok0, T0, tree_out=tree_out, verify_out=ver_out)
    dec_fig = decoder_layer_figure(w, dev, tree_out, rank)

    peak, peak_kind = hbm_peak()
    tpeak, tpeak_kind = tensor_peak()
    if dec_fig is not None:
        dec_fig["frac_of_hbm"] = dec_fig["achieved_gbs"] / peak
    achieved = gemm_bytes / (gemm_ms * 1e-3) / 1e9 if gemm_ms > 0 else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.is_bf16 else "f32",
        "data": "synthetic (seeded); target logits = the draft's logits of every tree node + "
                f"N(0, {w.target_sigma})",
        "config": dict(workload_config(w),
                       mode="eager launches through the C ABI from Python; CUDA events on the "
                            "launching stream"),
        "tree_nodes_per_s": value * B * n,
        "mean_accept_len": float(np.mean(accept)),
        "roofline": {"bound": "hbm", "kernel": "linear_bf16_tc_kernel (FC and LM head)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": None if achieved is None else achieved / peak,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": recorded_traffic(),
                     "algorithmic_bytes_per_launch": gemm_bytes / max(n_prof, 1),
                     "launches_timed": n_prof, "ms_per_launch": gemm_ms / max(n_prof, 1),
                     "timed_steps": f"GEMM launches of 1 step in {PROFILE_EVERY} (events stop "
                                    "those launches overlapping their predecessor)",
                     "gemm_ms_per_step_standalone": gemm_ms / max(len(sampled), 1),
                     "per_level": per_level(plist, peak, tpeak),
                     "tensor_peak": tpeak,
                     "tensor_peak_source": f"{tpeak_kind} bf16_tflops_sustained"},
        "clocks": clocks.summary(),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "eagle_tree_step_host per step: pinned host inputs and target logits "
                       "copied in, tree and verify results copied out, stream synchronised"},
        "gpu_launches": int(ranks.sum(launches)),
        "round_with_extend": {"value": 1e3 / round_ms, "unit": "rounds/s", "ms_per_round": round_ms,
                              "rounds": ROUNDS,
                              "how": "eagle_draft_extend from the previous verify (FC over every "
                                     "verified position + the next tree's level 0), levels 1..d-1, "
                                     "rerank/build, greedy verify; CUDA events, eager launches"},
        "static_tree": {"value": 1e3 / static_ms, "unit": "steps/s", "ms_per_step": static_ms,
                        "drafted_nodes": len(spec), "depth": d, "shape": "widths " + str(static_widths(d, w.topk)),
                        "how": "eagle_tree_init_static handle on the same weights: levels, build, greedy "
                               "verify against N(0,1) target logits; CUDA events, eager launches"},
        "sampling_verify": {"us_per_call": sample_us, "mean_accept_len": sample_accept,
                            "temperature": 1.0, "mode": "recursive rejection sampling",
                            "how": "eagle_verify_sample on the step's tree; q = draft logits of "
                                   "every node, p = the synthetic target; CUDA events, "
                                   f"{S_CALLS} calls"},
        "draft_decoder_layer": dec_fig,
        "greedy_verify": {"us_per_call": greedy_us, "target_logit_bytes": greedy_bytes,
                          "achieved_gbs": greedy_bytes / (greedy_us * 1e-6) / 1e9,
                          "frac_of_hbm": greedy_bytes / (greedy_us * 1e-6) / 1e9 / peak,
                          "target_logits_in_l2": in_l2,
                          "how": "eagle_verify_greedy (arg-max over the B x (m+1) x V target logits, "
                                 "then the walk) on the step's tree, alone; CUDA events, "
                                 f"{G_CALLS} calls over {N_INPUT_SETS} target sets; bytes = the "
                                 "target logits read"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    eng.close()
    ranks.close()


def main():
    args = parse_args()
    from eagle_speculative_decoding_draft_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_eagle(args, w)


if __name__ == "__main__":
    main()
