"""Seeded synthetic inputs for the mixture-of-experts layer workloads.

This module is the only code shared by the oracle side (tests, the CPU
baseline) and the CUDA side (tests, bench).  It holds no arithmetic of the
layer: it only draws random tensors and describes the workload shapes.

Workload shapes are the model shapes the "Mixture-of-Kittens" wiki page lists
under Key claims ("Validated on real frontier model shapes"), plus a tiny
case.  Recipe (one generator per tensor, reproducible on one device type):

* router logits: fp32 N(0, 1) [T, E], plus a per-expert bias:
  "zipf"  bias_e = 1.0 * ln((e + 1) ** -1.1)  (Zipf s = 1.1 rank weights),
  "hot8"  +3.0 on 8 experts drawn with numpy default_rng(seed);
* x: N(0, 1) drawn in fp32 and rounded to bf16 (round-to-nearest-even);
* expert e: W_gu [2m, d] ~ N(0, 1/d), W_dn [d, m] ~ N(0, 1/m), bf16, each
  expert from its own seeded generator so a single expert can be redrawn;
* shared expert: Ws_gu [2m_s, d] ~ N(0, 1/d), Ws_dn [d, m_s] ~ N(0, 1/m_s);
* output gradient dy: N(0, 1) bf16.
"""
import math

import numpy as np
import torch

# name -> shape and structure.  "fmt" is the routed experts' arithmetic.
WORKLOADS = {
    "tiny":            dict(T=256, d=256, m=128, E=8, k=2, m_shared=0, fmt="bf16", bias="none", seed=0, backward=True),
    "qwen3.5-397b":    dict(T=8192, d=4096, m=1024, E=512, k=10, m_shared=1024, fmt="bf16", bias="none", seed=1, backward=False),
    "glm-5.2":         dict(T=16384, d=6144, m=2048, E=256, k=8, m_shared=0, fmt="mxfp8", bias="zipf", seed=2, backward=False),
    "kimi-k2.7":       dict(T=16384, d=7168, m=2048, E=384, k=8, m_shared=2048, fmt="mxfp8", bias="zipf", seed=3, backward=True),
    "deepseek-v4-pro": dict(T=32768, d=7168, m=3072, E=384, k=6, m_shared=0, fmt="mxfp8", bias="hot8", seed=4, backward=False),
}
ORDER = ["tiny", "qwen3.5-397b", "glm-5.2", "kimi-k2.7", "deepseek-v4-pro"]

# Reduced-size variants with the same structure (routing skew, k, shared
# expert, format) that the oracle evaluates whole in seconds.  Sizes span
# several GEMM tiles and leave ragged tails (T not a multiple of 128, expert
# loads not multiples of 128, empty experts under skew).
SMALL = {
    "tiny":            dict(WORKLOADS["tiny"]),
    "qwen3.5-397b":    dict(T=300, d=512, m=256, E=24, k=10, m_shared=256, fmt="bf16", bias="none", seed=11, backward=False),
    "glm-5.2":         dict(T=520, d=768, m=256, E=32, k=8, m_shared=0, fmt="mxfp8", bias="zipf", seed=12, backward=False),
    "kimi-k2.7":       dict(T=392, d=512, m=256, E=40, k=8, m_shared=256, fmt="mxfp8", bias="zipf", seed=13, backward=True),
    "deepseek-v4-pro": dict(T=1000, d=512, m=384, E=48, k=6, m_shared=0, fmt="mxfp8", bias="hot8", seed=14, backward=False),
}


def _seed(*parts):
    h = 1469598103934665603
    for p in parts:
        for ch in str(p).encode():
            h = ((h ^ ch) * 1099511628211) % (1 << 63)
        h = ((h ^ 0xFF) * 1099511628211) % (1 << 63)
    return h


def _gen(device, *parts):
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def _normal(shape, std, device, *parts):
    t = torch.randn(shape, generator=_gen(device, *parts), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def router_bias(cfg):
    E = cfg["E"]
    b = np.zeros(E, dtype=np.float32)
    if cfg["bias"] == "zipf":
        b = (1.0 * np.log((np.arange(E, dtype=np.float64) + 1.0) ** -1.1)).astype(np.float32)
    elif cfg["bias"] == "hot8":
        hot = np.random.default_rng(cfg["seed"]).choice(E, size=8, replace=False)
        b[hot] += np.float32(3.0)
    return b


def logits(cfg, device="cpu"):
    l = _normal((cfg["T"], cfg["E"]), 1.0, device, cfg["seed"], "logits")
    return l + torch.from_numpy(router_bias(cfg)).to(device)


def tokens(cfg, device="cpu"):
    return _normal((cfg["T"], cfg["d"]), 1.0, device, cfg["seed"], "x").to(torch.bfloat16)


def expert(cfg, e, device="cpu"):
    """(W_gu [2m, d], W_dn [d, m]) bf16 of expert e."""
    d, m = cfg["d"], cfg["m"]
    gu = _normal((2 * m, d), 1.0 / math.sqrt(d), device, cfg["seed"], "gu", e).to(torch.bfloat16)
    dn = _normal((d, m), 1.0 / math.sqrt(m), device, cfg["seed"], "dn", e).to(torch.bfloat16)
    return gu, dn


def experts(cfg, device="cpu"):
    """Stacked (W_gu [E, 2m, d], W_dn [E, d, m]) bf16."""
    E, d, m = cfg["E"], cfg["d"], cfg["m"]
    gu = torch.empty((E, 2 * m, d), dtype=torch.bfloat16, device=device)
    dn = torch.empty((E, d, m), dtype=torch.bfloat16, device=device)
    for e in range(E):
        gu[e], dn[e] = expert(cfg, e, device)
    return gu, dn


def shared(cfg, device="cpu"):
    """(Ws_gu [2m_s, d], Ws_dn [d, m_s]) bf16, or None."""
    ms, d = cfg["m_shared"], cfg["d"]
    if not ms:
        return None
    gu = _normal((2 * ms, d), 1.0 / math.sqrt(d), device, cfg["seed"], "s_gu").to(torch.bfloat16)
    dn = _normal((d, ms), 1.0 / math.sqrt(ms), device, cfg["seed"], "s_dn").to(torch.bfloat16)
    return gu, dn


def out_grad(cfg, device="cpu"):
    return _normal((cfg["T"], cfg["d"]), 1.0, device, cfg["seed"], "dy").to(torch.bfloat16)


def sample_tokens(cfg, n=256):
    """Seeded subset of token indices (sorted) used where the oracle cannot run whole."""
    rng = np.random.default_rng(cfg["seed"] + 1000)
    return np.sort(rng.choice(cfg["T"], size=min(n, cfg["T"]), replace=False))


def sample_experts(counts, seed, n=4, max_rows=None):
    """Seeded choice of n experts with at least one routed row (optionally capped load)."""
    counts = np.asarray(counts)
    ok = np.nonzero((counts > 0) & ((counts <= max_rows) if max_rows else True))[0]
    rng = np.random.default_rng(seed + 2000)
    return np.sort(rng.choice(ok, size=min(n, ok.size), replace=False))


def to_f64(t):
    """float64 numpy copy of a (bf16 / fp32) torch tensor on any device."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)
