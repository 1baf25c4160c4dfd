"""The dispatch ring: the forward's dispatch and gate/up GEMM as one persistent
launch in which gather SMs fill a fixed ring of 128-row tiles that the GEMM SMs
consume.  The GEMM sees the same codes in the same order as with the
materialised dispatch, so every output must be bitwise identical for every ring
size and SM split, including rings far smaller than one expert's rows (the
hot experts of the DeepSeek-V4-Pro shape pass through in pieces)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import TOL, Case, rel

pytestmark = pytest.mark.gpu

RINGS = [(128, 1), (384, 3), (1024, 8)]   # (ring_rows, gather SMs)


def with_ring(L, ring_rows, gather_sms, flags=None):
    import mixture_experts_layer_device_gb300 as pkg
    c = L.cfg
    return pkg.MoeConfig(c.T, c.d, c.m, c.E, c.k, c.m_shared, c.dtype, c.flags if flags is None else flags,
                         ring_rows, gather_sms)


def forward(L, cfg, x, lg, train):
    """One moe_forward on fresh zero-filled buffers: (y, saved, ws)."""
    import mixture_experts_layer_device_gb300 as pkg
    ws = torch.zeros(pkg.moe_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    saved = torch.zeros(pkg.moe_saved_bytes(cfg), dtype=torch.uint8, device="cuda") if train else None
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    pkg.check(pkg.moe_forward(cfg, x, lg, L.W, y, saved, ws))
    assert pkg.moe_get_status(ws) == 0
    return y, saved, ws


def buf(cfg, base, which, name):
    import mixture_experts_layer_device_gb300 as pkg
    off, nb = pkg.moe_buffer_info(cfg, which, name)
    return base[off:off + nb]


@pytest.mark.parametrize("name", ["glm-5.2", "kimi-k2.7", "deepseek-v4-pro"])
@pytest.mark.parametrize("ring_rows,gather_sms", RINGS)
def test_ring_forward_bitwise_equal(name, ring_rows, gather_sms):
    cfg = dict(mi.SMALL[name])
    c = Case(cfg, backward=True)
    L = c.layer
    y0, s0, w0 = forward(L, with_ring(L, 0, 0), c.xg, c.lg, train=False)
    rc = with_ring(L, ring_rows, gather_sms)
    y1, s1, w1 = forward(L, rc, c.xg, c.lg, train=False)
    assert torch.equal(y0, y1)
    assert torch.equal(buf(L.cfg, w0, 1, "hq"), buf(rc, w1, 1, "hq"))
    assert torch.equal(buf(L.cfg, w0, 1, "hq_sf"), buf(rc, w1, 1, "hq_sf"))
    # training forward: every saved activation (incl. the column-blocked x codes)
    y0, s0, _ = forward(L, with_ring(L, 0, 0), c.xg, c.lg, train=True)
    y1, s1, _ = forward(L, rc, c.xg, c.lg, train=True)
    assert torch.equal(y0, y1)
    assert torch.equal(s0, s1)


def test_ring_backward_bitwise_equal():
    import mixture_experts_layer_device_gb300 as pkg
    cfg = dict(mi.SMALL["kimi-k2.7"])
    c = Case(cfg, backward=True)
    L = c.layer
    grads = []
    for rr, gs in [(0, 0), (256, 2)]:
        rc = with_ring(L, rr, gs)
        y, saved, ws = forward(L, rc, c.xg, c.lg, train=True)
        g = L.alloc_grads()
        pkg.check(pkg.moe_backward(rc, c.dyg, c.xg, L.W, saved, g["dx"], g["dlogits"], g["dW_gu"], g["dW_dn"],
                                   g["dWs_gu"], g["dWs_dn"], ws))
        assert pkg.moe_get_status(ws) == 0
        grads.append(g)
    for n in ("dx", "dlogits", "dW_gu", "dW_dn", "dWs_gu", "dWs_dn"):
        assert torch.equal(grads[0][n], grads[1][n]), n


def test_ring_forward_matches_oracle():
    """A one-slot ring with one gather SM: the most serialised hand-off."""
    cfg = dict(mi.SMALL["deepseek-v4-pro"])
    c = Case(cfg, backward=False)
    L = c.layer
    y, _, _ = forward(L, with_ring(L, 128, 1), c.xg, c.lg, train=False)
    y_ref, _ = c.oracle_forward()
    assert rel(mi.to_f64(y), y_ref) < TOL[cfg["fmt"]]


def test_ring_timeout_reported_and_context_survives():
    """With the debug flag the gather SMs publish nothing: the GEMM SMs' ring
    waits run out (50 ms), the call returns with MOE_ERR_TIMEOUT, and the next
    call on the same workspace is correct."""
    import time
    import mixture_experts_layer_device_gb300 as pkg
    cfg = dict(mi.SMALL["deepseek-v4-pro"])
    c = Case(cfg, backward=False)
    L = c.layer
    starve = with_ring(L, 256, 2, flags=L.cfg.flags | pkg.MOE_FLAG_DEBUG_STARVE)
    ring = with_ring(L, 256, 2)
    ws = torch.zeros(pkg.moe_workspace_bytes(ring), dtype=torch.uint8, device="cuda")
    y = torch.empty((cfg["T"], cfg["d"]), dtype=torch.bfloat16, device="cuda")
    t0 = time.time()
    pkg.check(pkg.moe_forward(starve, c.xg, c.lg, L.W, y, None, ws))
    assert pkg.moe_get_status(ws) == -6
    assert time.time() - t0 < 30
    pkg.check(pkg.moe_forward(ring, c.xg, c.lg, L.W, y, None, ws))
    assert pkg.moe_get_status(ws) == 0
    y_ref, _ = c.oracle_forward()
    assert rel(mi.to_f64(y), y_ref) < TOL[cfg["fmt"]]
