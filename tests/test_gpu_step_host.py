"""The host-buffer step (eagle_tree_step_host) against the device-resident step: same kernels,
so every output must agree bit for bit; repeated calls (staging reused), positions given or not,
the mask optional, and the status word returned clean."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_draft_gb300 import synth
from parity import to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("wl,tdt", [(1, "f32"), (2, "f32"), (2, "bf16")])
def test_host_step_matches_the_device_step(dev, wl, tdt):
    from eagle_speculative_decoding_draft_gb300.engine import EagleTree
    w = synth.WORKLOADS[wl]
    inp = synth.make_inputs(w)
    g = lambda t: t.to(dev).contiguous()
    eng = EagleTree(g(inp.w_fc), g(inp.b_fc) if w.bias else None, g(inp.w_lm), g(inp.emb),
                    w.batch, w.depth, w.topk, w.num_keep)
    B, n, d, W = w.batch, w.num_nodes, w.depth, eng.mask_words
    rng = np.random.default_rng(wl)
    i32 = dict(dtype=torch.int32, pin_memory=True)
    staging = None
    for it in range(3):
        if it == 0:
            feat, tok = inp.root_feat, inp.root_tok
        else:
            fdt = torch.bfloat16 if w.is_bf16 else torch.float32
            feat = torch.from_numpy(rng.standard_normal((B, w.hidden), dtype=np.float32)).to(fdt)
            tok = torch.from_numpy(rng.integers(0, w.vocab, size=B).astype(np.int32))
        pos = torch.from_numpy(rng.integers(0, 1000, size=B).astype(np.int32)) if it != 1 else None
        fd, td = g(feat), g(tok)
        tree = eng.draft(fd, td, None if pos is None else g(pos))
        nz = eng.node_logits(fd)
        T = (nz + torch.randn(nz.shape, device=dev, generator=torch.Generator(device=dev).manual_seed(it))).contiguous()
        if tdt == "bf16":  # the target logits a bf16 target model emits
            T = T.to(torch.bfloat16)
        ver = eng.verify_greedy(tree["tokens"], tree["parents"], T)
        torch.cuda.synchronize()
        if staging is None:
            staging = torch.empty_like(T)
        host = {"tokens": torch.empty(B, n, **i32), "parents": torch.empty(B, n, **i32),
                "positions": torch.empty(B, n, **i32), "accept_len": torch.empty(B, **i32),
                "accept_tokens": torch.empty(B, d + 1, **i32)}
        if it != 2:
            host["mask"] = torch.empty(B, n, W, **i32)
        eng.step_host(feat.pin_memory(), tok.pin_memory(), T.cpu().pin_memory(), staging, host,
                      pos_base=None if pos is None else pos.pin_memory())
        assert torch.equal(host["tokens"], tree["tokens"].cpu())
        assert torch.equal(host["parents"], tree["parents"].cpu())
        assert torch.equal(host["positions"], tree["positions"].cpu())
        if "mask" in host:
            assert torch.equal(host["mask"], tree["mask"].cpu())
        assert torch.equal(host["accept_len"], ver["accept_len"].cpu())
        assert torch.equal(host["accept_tokens"], ver["accept_tokens"].cpu())
        assert torch.equal(staging.cpu(), T.cpu())
        # every call after the first capture replays the graph
        if it >= 1:
            assert eng.step_graphed() == 1
    eng.status()
    eng.close()
