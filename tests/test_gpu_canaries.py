"""Guard words around every buffer the draft-tree step writes.

Each output (the tree arrays, the mask, the scores, the verify results, the per-level logits, the
node logits, the draft-extend outputs) and the handle's workspace is a slice of a larger buffer
whose 4 KB on either side hold a known byte pattern; after the step the pattern must be intact,
so no kernel writes outside what it was given.  It runs on the regular build here and on the
checking build (-DEAGLE_CHECKS) through tests/test_gpu_checks.py."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_draft_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0x5A


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from eagle_speculative_decoding_draft_gb300 import build, _lib
    build.build()
    _lib.load()
    return torch.device("cuda:0")


class Guarded:
    """Tensors carved out of guard-padded byte buffers."""

    def __init__(self, dev):
        self.dev = dev
        self.bufs = []

    def empty(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        raw = torch.full((GUARD + ((n + 255) // 256) * 256 + GUARD,), PATTERN, dtype=torch.uint8, device=self.dev)
        self.bufs.append((raw, n))
        return raw[GUARD:GUARD + n].view(dtype).view(*shape)

    def check(self):
        torch.cuda.synchronize()
        for raw, n in self.bufs:
            host = raw.cpu().numpy()
            assert np.all(host[:GUARD] == PATTERN), "write before a buffer"
            assert np.all(host[GUARD + n:] == PATTERN), "write after a buffer"


@pytest.mark.parametrize("case", [dict(h=64, V=1000, B=20, d=4, k=4, m=15, dtype="bf16"),
                                  dict(h=96, V=3000, B=3, d=5, k=10, m=60, dtype="bf16"),
                                  dict(h=32, V=300, B=3, d=4, k=3, m=12, dtype="f32")],
                         ids=lambda c: "h{h}V{V}B{B}d{d}k{k}m{m}{dtype}".format(**c))
def test_every_output_stays_inside_its_buffer(dev, case):
    from eagle_speculative_decoding_draft_gb300.engine import EagleTree
    w = synth.custom(case["h"], case["V"], case["B"], case["d"], case["k"], case["m"], dtype=case["dtype"])
    inp = synth.make_inputs(w, seed=7)
    g = lambda t: t.to(dev).contiguous()
    G = Guarded(dev)
    probe = EagleTree(g(inp.w_fc), g(inp.b_fc), g(inp.w_lm), g(inp.emb), w.batch, w.depth, w.topk, w.num_keep)
    nbytes = probe.workspace.numel()
    probe.close()
    ws = G.empty((nbytes,), torch.uint8)
    eng = EagleTree(g(inp.w_fc), g(inp.b_fc), g(inp.w_lm), g(inp.emb), w.batch, w.depth, w.topk, w.num_keep,
                    workspace=ws)
    B, n, d, V, W = w.batch, w.num_nodes, w.depth, w.vocab, eng.mask_words
    i32 = torch.int32
    tree = {"tokens": G.empty((B, n), i32), "parents": G.empty((B, n), i32), "positions": G.empty((B, n), i32),
            "mask": G.empty((B, n, W), i32), "logscore": G.empty((B, n), torch.float32)}
    ver = {"accept_len": G.empty((B,), i32), "accept_nodes": G.empty((B, d + 1), i32),
           "accept_tokens": G.empty((B, d + 1), i32)}
    logits = G.empty((d, B * w.topk, V), torch.float32)
    pos = g(torch.arange(B, dtype=torch.int32) * 3)
    feat, tok = g(inp.root_feat), g(inp.root_tok)
    eng.draft(feat, tok, pos, tree_out=tree, logits_out=logits)
    nz = eng.node_logits(feat, out=G.empty((B, n, V), torch.float32))
    T = (nz + 0.5).contiguous()
    eng.verify_greedy(tree["tokens"], tree["parents"], T, out=ver)
    # the next round through draft extend
    fdt = torch.bfloat16 if w.is_bf16 else torch.float32
    F = g(torch.randn(B, n, w.hidden).to(fdt))
    eng.extend(F, ver["accept_len"], ver["accept_nodes"], ver["accept_tokens"],
               path_fhat=G.empty((B, d + 1, w.hidden), fdt))
    for lvl in range(1, d):
        eng.draft_level(lvl)
    eng.rerank_build_tree(pos, out=tree)
    eng.status()
    G.check()
    eng.close()
