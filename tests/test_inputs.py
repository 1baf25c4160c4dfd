"""The seeded synthetic inputs, on CPU: shapes, determinism, the weight scales
and router biases of the recipe, and the load structure each full-size
workload's routing must have (Zipf-skewed, 8 hot experts, near-uniform).  The
load bands bracket figures worked out independently from the workload
definitions; any draw of the recipe lands inside them."""
import math

import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe as om


def test_draws_are_seeded_and_shaped():
    cfg = mi.SMALL["kimi-k2.7"]
    T, d, m, E, ms = cfg["T"], cfg["d"], cfg["m"], cfg["E"], cfg["m_shared"]
    x, l, dy = mi.tokens(cfg), mi.logits(cfg), mi.out_grad(cfg)
    assert x.shape == (T, d) and x.dtype == torch.bfloat16
    assert l.shape == (T, E) and l.dtype == torch.float32
    assert dy.shape == (T, d) and dy.dtype == torch.bfloat16
    gu, dn = mi.experts(cfg)
    assert gu.shape == (E, 2 * m, d) and dn.shape == (E, d, m) and gu.dtype == torch.bfloat16
    sgu, sdn = mi.shared(cfg)
    assert sgu.shape == (2 * ms, d) and sdn.shape == (d, ms)
    assert torch.equal(mi.tokens(cfg), x) and torch.equal(mi.logits(cfg), l)
    assert torch.equal(mi.expert(cfg, 3)[0], gu[3])         # one expert re-drawn alone
    assert not torch.equal(x, dy)                          # distinct streams per tensor
    assert not torch.equal(gu[0], gu[1])


def test_weight_scales():
    cfg = dict(mi.SMALL["kimi-k2.7"])
    gu, dn = mi.expert(cfg, 0)
    d, m = cfg["d"], cfg["m"]
    assert gu.float().std().item() == pytest.approx(1 / math.sqrt(d), rel=0.03)
    assert dn.float().std().item() == pytest.approx(1 / math.sqrt(m), rel=0.03)
    x = mi.tokens(cfg).float()
    assert abs(x.mean().item()) < 0.01 and x.std().item() == pytest.approx(1.0, rel=0.02)


def test_router_biases():
    z = mi.router_bias(dict(E=6, bias="zipf", seed=0))
    assert z.dtype == np.float32 and z[0] == 0.0
    assert np.allclose(z, -1.1 * np.log(np.arange(1, 7)), rtol=1e-6)
    assert np.all(np.diff(z) < 0)
    h = mi.router_bias(dict(E=384, bias="hot8", seed=4))
    assert np.count_nonzero(h) == 8 and np.all(h[h != 0] == 3.0)
    assert np.array_equal(h, mi.router_bias(dict(E=384, bias="hot8", seed=4)))
    assert not np.any(mi.router_bias(dict(E=7, bias="none", seed=0)))


def _counts(name):
    cfg = mi.WORKLOADS[name]
    idx, _ = om.route(mi.logits(cfg).numpy(), cfg["k"])
    return cfg, idx, np.bincount(idx.reshape(-1), minlength=cfg["E"])


@pytest.mark.parametrize("name,empty_band", [("glm-5.2", (25, 60)), ("kimi-k2.7", (120, 190))])
def test_zipf_workloads_pile_onto_the_first_experts(name, empty_band):
    cfg, idx, cnt = _counts(name)
    T = cfg["T"]
    assert cnt.argmax() == 0 and 0.9 * T < cnt[0] <= T      # nearly every token picks expert 0
    assert (idx == 0).any(axis=1).mean() > 0.95
    assert empty_band[0] <= np.count_nonzero(cnt == 0) <= empty_band[1]


def test_hot8_workload_has_eight_dominant_experts():
    cfg, _, cnt = _counts("deepseek-v4-pro")
    hot = np.nonzero(mi.router_bias(cfg))[0]
    mean = cfg["T"] * cfg["k"] / cfg["E"]
    assert np.all((cnt[hot] > 35 * mean) & (cnt[hot] < 42 * mean))   # about 19.8k rows each
    cold = np.delete(cnt, hot)
    assert 80 < cold.mean() < 130


def test_unbiased_workload_is_near_uniform():
    cfg, _, cnt = _counts("qwen3.5-397b")
    mean = cfg["T"] * cfg["k"] / cfg["E"]
    assert np.count_nonzero(cnt == 0) == 0
    assert cnt.max() < 1.5 * mean and cnt.min() > 0.5 * mean
