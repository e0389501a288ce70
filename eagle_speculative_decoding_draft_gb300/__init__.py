"""GB300 (sm_103a) EAGLE / EAGLE-2 dynamic draft-tree engine.

The hot path (draft FC + LM head on tcgen05 tensor cores, per-row log-softmax/top-k, expand,
rerank, tree build, greedy verify) runs in hand-written CUDA kernels behind the C ABI of
include/eagle_tree.h; ``engine`` marshals torch tensors into it.
"""
from . import synth  # noqa: F401  (seeded inputs; no method arithmetic)


def __getattr__(name):
    if name in ("EagleTree", "row_topk", "expand", "build_tree", "verify_walk", "linear_bf16"):
        from . import engine
        return getattr(engine, name)
    raise AttributeError(name)
