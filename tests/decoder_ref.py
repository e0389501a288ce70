"""Shared pieces of the draft decoder layer tests: seeded bf16 weights and inputs, the ancestor
mask of a parent list, and a float64 torch restatement of the layer (library attention, no
intermediate rounding) with the first-order size of its bf16 rounding terms."""
import numpy as np
import torch


def bf(*shape, s=0.1, g=None):
    return (torch.randn(*shape, generator=g) * s).to(torch.bfloat16)


def layer(B=2, n=5, P=4, h=64, H=4, Hk=2, D=16, I=48, seed=0, norm_ones=False, fan_in=False):
    """Seeded layer inputs.  fan_in: weight std 1/sqrt(fan-in) (Llama-style init, for large h);
    else the fixed small-size scales."""
    g = torch.Generator().manual_seed(seed)
    sd = (lambda k, s: k ** -0.5) if fan_in else (lambda k, s: s)
    w = dict(x=bf(B, n, h, s=1.0, g=g), w_qkv=bf((H + 2 * Hk) * D, h, s=sd(h, 0.15), g=g),
             w_o=bf(h, H * D, s=sd(H * D, 0.1), g=g),
             w_norm=(torch.ones(h) if norm_ones else 1 + 0.1 * torch.randn(h, generator=g)).to(torch.bfloat16),
             w_gu=bf(2 * I, h, s=sd(h, 0.1), g=g), w_d=bf(h, I, s=sd(I, 0.1), g=g),
             k_cache=bf(B, P, Hk, D, s=1.0, g=g), v_cache=bf(B, P, Hk, D, s=1.0, g=g))
    return w, dict(B=B, n=n, P=P, h=h, H=H, Hk=Hk, D=D, I=I)


def random_tree(n, max_depth, rng):
    """parents (parent before child) and depths of an n-node tree rooted at node 0."""
    parents, depths = [-1], [0]
    for i in range(1, n):
        cand = [j for j in range(i) if depths[j] < max_depth]
        p = int(cand[rng.integers(0, len(cand))])
        parents.append(p)
        depths.append(depths[p] + 1)
    return parents, depths


def tolerance(h1, ref, absterms):
    """First-order size of the layer's bf16 rounding points: half an ulp (2^-8 relative, doubled for
    margin) of each residual sum, and of the rounded attention output and MLP product carried
    through the output and down projections (their sums of absolute terms)."""
    return 2.0 ** -7 * (np.abs(h1) + np.abs(ref)) + 2.0 ** -6 * absterms + 1e-4


def tree_mask(parents):
    n = len(parents)
    W = (n + 31) // 32
    m = np.zeros((n, W), np.uint32)
    for i in range(n):
        x = i
        while x >= 0:
            m[i, x // 32] |= np.uint32(1 << (x % 32))
            x = parents[x]
    return m


def rope64(x, pos, theta=10000.0):
    D = x.shape[-1]
    half = D // 2
    j = torch.arange(half, dtype=torch.float64)
    ang = pos[..., None].double() * theta ** (-2 * j / D)
    c, s = torch.cos(ang), torch.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return torch.cat([a * c - b * s, b * c + a * s], dim=-1)


def reference_layer(w, d, parents, pos):
    """float64 torch restatement (library attention), no intermediate rounding.  Returns the
    layer output, h1 and the sums of absolute terms of the output and down projections."""
    B, n, P, h, H, Hk, D, I = (d[k] for k in ("B", "n", "P", "h", "H", "Hk", "D", "I"))
    f = lambda t: t.double()
    x = f(w["x"])
    qkv = x @ f(w["w_qkv"]).T
    q = qkv[..., :H * D].reshape(B, n, H, D)
    k = qkv[..., H * D:(H + Hk) * D].reshape(B, n, Hk, D)
    v = qkv[..., (H + Hk) * D:].reshape(B, n, Hk, D)
    pos = torch.as_tensor(np.asarray(pos), dtype=torch.int64)
    q = rope64(q, pos[..., None].expand(B, n, H))
    k = rope64(k, pos[..., None].expand(B, n, Hk))
    K = torch.cat([f(w["k_cache"]), k], dim=1)
    Vv = torch.cat([f(w["v_cache"]), v], dim=1)
    rep = H // Hk
    K = K.repeat_interleave(rep, dim=2).permute(0, 2, 1, 3)
    Vv = Vv.repeat_interleave(rep, dim=2).permute(0, 2, 1, 3)
    allow = torch.zeros(n, P + n, dtype=torch.bool)
    allow[:, :P] = True
    for i in range(n):
        x_ = i
        while x_ >= 0:
            allow[i, P + x_] = True
            x_ = parents[x_]
    o = torch.nn.functional.scaled_dot_product_attention(q.permute(0, 2, 1, 3), K, Vv, attn_mask=allow)
    o = o.permute(0, 2, 1, 3).reshape(B, n, H * D)
    h1 = x + o @ f(w["w_o"]).T
    abs_o = o.abs() @ f(w["w_o"]).abs().T
    r = h1 / torch.sqrt((h1 * h1).mean(-1, keepdim=True) + 1e-6) * f(w["w_norm"])
    gu = r @ f(w["w_gu"]).T
    g_, u = gu[..., :I], gu[..., I:]
    a = torch.nn.functional.silu(g_) * u
    abs_d = a.abs() @ f(w["w_d"]).abs().T
    return (h1 + a @ f(w["w_d"]).T).numpy(), h1.numpy(), (abs_o + abs_d).numpy()
