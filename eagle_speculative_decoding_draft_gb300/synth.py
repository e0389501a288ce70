"""Seeded synthetic inputs for the draft-tree workloads.

This module only draws random numbers in the shapes and distributions of the five workloads;
it holds none of the method's arithmetic.  It is the one piece of code that both the CUDA
path's callers and the CPU oracle's callers consume.

Distributions (normal parameters are (mean, standard deviation)):
  W_fc [h][2h] ~ N(0, 1/sqrt(2h))      FC weight
  b_fc [h]     ~ N(0, 0.02), or 0       FC bias (zero for the tiny and the SGLang-default shape)
  W_lm [V][h]  ~ N(0, 3/sqrt(h))        shared frozen LM head
  E    [V][h]  ~ N(0, 0.02)             shared frozen token embedding
  f    [B][h]  ~ N(0, 1)                the target's feature at the root
  root [B]     ~ U{0..V-1}              the root (last committed) token
  noise         ~ N(0, sigma)           added to draft logits to make target logits
Values are drawn in fp32 from numpy's PCG64 stream seeded with 1000 + workload number, in the
order above, then rounded to bf16 (round to nearest even, by torch) for bf16 workloads.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    number: int          # 0 for custom shapes
    name: str
    dtype: str           # "f32" or "bf16": weights, embedding and features
    hidden: int          # h
    vocab: int           # V
    batch: int           # B
    depth: int           # d: drafted levels
    topk: int            # k
    num_keep: int        # m: drafted nodes kept (tree has m+1 nodes with the root)
    bias: bool           # FC bias drawn (else zero)
    target_sigma: float  # std of the noise added to draft logits to form target logits

    @property
    def is_bf16(self) -> bool:
        return self.dtype == "bf16"

    @property
    def num_candidates(self) -> int:
        return self.topk + (self.depth - 1) * self.topk * self.topk

    @property
    def num_nodes(self) -> int:
        return self.num_keep + 1

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    1: Workload(1, "tiny-fp32 h256 V1024 B1 d3 k2 m6", "f32", 256, 1024, 1, 3, 2, 6, False, 1.0),
    2: Workload(2, "vicuna7b-shape h4096 V32000 B1 d6 k10 m60", "bf16", 4096, 32000, 1, 6, 10, 60,
                True, 1.0),
    3: Workload(3, "sglang-default h4096 V32000 B64 d5 k4 m7", "bf16", 4096, 32000, 64, 5, 4, 7,
                False, 0.5),
    4: Workload(4, "llama2-70b-shape h8192 V32000 B4 d6 k10 m48", "bf16", 8192, 32000, 4, 6, 10,
                48, True, 1.5),
    5: Workload(5, "llama3-8b-vocab h4096 V128256 B32 d5 k8 m64", "bf16", 4096, 128256, 32, 5, 8,
                64, True, 1.0),
}


def custom(hidden, vocab, batch, depth, topk, num_keep, dtype="bf16", bias=True,
           target_sigma=1.0, name="custom") -> Workload:
    return Workload(0, name, dtype, hidden, vocab, batch, depth, topk, num_keep, bias,
                    target_sigma)


@dataclass
class Inputs:
    workload: Workload
    w_fc: torch.Tensor      # [h][2h]
    b_fc: torch.Tensor      # [h]
    w_lm: torch.Tensor      # [V][h]
    emb: torch.Tensor       # [V][h]
    root_feat: torch.Tensor  # [B][h]
    root_tok: torch.Tensor   # [B] int32
    rng: np.random.Generator  # continues the stream (target noise is drawn from it)


def _normal(rng, shape, std, dtype):
    a = rng.standard_normal(shape, dtype=np.float32)
    a *= np.float32(std)
    t = torch.from_numpy(a)
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def make_inputs(w: Workload, seed: int | None = None) -> Inputs:
    """Draw one workload's weights and root inputs (CPU tensors)."""
    rng = np.random.default_rng(1000 + w.number if seed is None else seed)
    h, V, B = w.hidden, w.vocab, w.batch
    w_fc = _normal(rng, (h, 2 * h), 1.0 / np.sqrt(2.0 * h), w.dtype)
    if w.bias:
        b_fc = _normal(rng, (h,), 0.02, w.dtype)
    else:
        b_fc = torch.zeros(h, dtype=torch.bfloat16 if w.is_bf16 else torch.float32)
    w_lm = _normal(rng, (V, h), 3.0 / np.sqrt(h), w.dtype)
    emb = _normal(rng, (V, h), 0.02, w.dtype)
    root_feat = _normal(rng, (B, h), 1.0, w.dtype)
    root_tok = torch.from_numpy(rng.integers(0, V, size=B, dtype=np.int64).astype(np.int32))
    return Inputs(w, w_fc, b_fc, w_lm, emb, root_feat, root_tok, rng)


def extra_roots(w: Workload, count: int, seed: int):
    """`count` more root inputs (features [count][h] ~ N(0, 1), tokens ~ U{0..V-1}) for the same
    weights, from their own seeded stream; returns CPU tensors (features in the workload's dtype,
    tokens int32)."""
    rng = np.random.default_rng(seed)
    feat = _normal(rng, (count, w.hidden), 1.0, w.dtype)
    tok = torch.from_numpy(rng.integers(0, w.vocab, size=count, dtype=np.int64).astype(np.int32))
    return feat, tok


def target_noise(inp: Inputs, shape=None) -> np.ndarray:
    """N(0, sigma) noise, float32, of shape [B][m+1][V] by default, drawn next in the stream."""
    w = inp.workload
    if shape is None:
        shape = (w.batch, w.num_nodes, w.vocab)
    a = inp.rng.standard_normal(shape, dtype=np.float32)
    a *= np.float32(w.target_sigma)
    return a
