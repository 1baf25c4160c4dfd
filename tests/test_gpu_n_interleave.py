"""The grouped-M GEMMs' interleaved tile order on a bimodal expert load.

When every active expert has either one or two 128-row tiles (light) or at
least 16 (heavy), the forward and dgrad GEMMs spread the light experts' tiles
among the heavy experts' tiles.  The order changes which CTA computes a tile
and when, never the arithmetic of a tile, so:

* the outputs match the oracle like the expert-ordered case;
* the forward's output equals, bit for bit, the ring path's, which keeps
  expert order (a fused dispatch cannot run ahead of its gather).

The case (T = 3000, E = 64, top-6, eight hot experts) is chosen so that the
load is bimodal; the test checks that on the oracle's routing first."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import TOL, Case, padded_rows, rel
from oracle import moe as om

pytestmark = pytest.mark.gpu

LIGHT_MTILES = 3   # fewer 128-row tiles than this: a light expert
HEAVY_MIN = 16     # every other active expert has at least this many


def bimodal_cfg(fmt):
    return dict(T=3000, d=512, m=384, E=64, k=6, m_shared=0, fmt=fmt, bias="hot8", seed=32, backward=True)


def assert_bimodal(counts):
    mt = (np.asarray(counts) + 127) // 128
    light = (mt > 0) & (mt < LIGHT_MTILES)
    heavy = mt >= LIGHT_MTILES
    assert light.any() and heavy.any() and mt[heavy].min() >= HEAVY_MIN, mt


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_forward_on_bimodal_load_matches_oracle(fmt):
    cfg = bimodal_cfg(fmt)
    c = Case(cfg, backward=True)
    y = c.layer.forward(c.xg, c.lg, train=True)
    assert c.layer.status() == 0
    y_ref, s = c.oracle_forward()
    assert_bimodal(s["counts"])
    counts, offsets, poff, _ = c.route_views(0)
    assert np.array_equal(counts, s["counts"])
    pr = padded_rows(counts, offsets, poff)
    L = c.layer
    n = int(poff[-1])
    GU = L.view(0, "GU", "bf16", (L.Rp, 2 * cfg["m"]))[:n].float().cpu().numpy().astype(np.float64)
    o = L.view(0, "o", "bf16", (L.Rp, cfg["d"]))[:n].float().cpu().numpy().astype(np.float64)
    tol = TOL[fmt]
    assert rel(GU[pr], s["GU"]) < tol, "gate/up GEMM"
    assert rel(o[pr], s["o"]) < tol, "down GEMM"
    yg = y.float().cpu().numpy()
    assert rel(yg, y_ref) < tol
    err = np.abs(yg - y_ref)
    assert err.max() <= 0.05 * np.abs(y_ref).max() + 1e-2
    # every light and heavy expert's rows: no expert's tiles were skipped or doubled
    for e in range(cfg["E"]):
        r0, r1 = int(s["offsets"][e]), int(s["offsets"][e + 1])
        if r1 > r0:
            assert rel(o[pr][r0:r1], s["o"][r0:r1]) < tol, "expert %d" % e


def test_backward_on_bimodal_load_matches_oracle():
    cfg = bimodal_cfg("mxfp8")
    c = Case(cfg, backward=True)
    c.layer.forward(c.xg, c.lg, train=True)
    grads = c.layer.alloc_grads()
    for v in grads.values():
        if v is not None:
            v.fill_(float("nan"))
    g = c.layer.backward(c.dyg, c.xg, grads=grads)
    assert c.layer.status() == 0
    _, saved = c.oracle_forward()
    assert_bimodal(saved["counts"])
    ref = om.backward(mi.to_f64(c.dy), mi.to_f64(c.x), c.oracle_experts(), cfg["k"], cfg["fmt"], saved)
    tol = TOL["mxfp8"]
    assert rel(g["dx"].float().cpu().numpy(), ref["dx"]) < tol, "dx"
    assert rel(g["dlogits"].cpu().numpy(), ref["dlogits"]) < tol, "dlogits"
    dW_gu = g["dW_gu"].float().cpu().numpy()
    dW_dn = g["dW_dn"].float().cpu().numpy()
    for e in range(cfg["E"]):
        assert rel(dW_gu[e], ref["dW_gu"][e]) < tol, "dW_gu[%d]" % e
        assert rel(dW_dn[e], ref["dW_dn"][e]) < tol, "dW_dn[%d]" % e


def test_interleaved_forward_bitwise_equals_expert_ordered_ring():
    import mixture_experts_layer_device_gb300 as pkg
    cfg = bimodal_cfg("mxfp8")
    c = Case(cfg, backward=False)
    y0 = c.layer.forward(c.xg, c.lg)
    assert c.layer.status() == 0
    counts = c.layer.view(1, "counts", "i32", (cfg["E"],)).cpu().numpy()
    assert_bimodal(counts)
    L = c.layer.cfg
    rc = pkg.MoeConfig(L.T, L.d, L.m, L.E, L.k, L.m_shared, L.dtype, L.flags, 1024, 4)
    ws = torch.empty(pkg.moe_workspace_bytes(rc), dtype=torch.uint8, device="cuda")
    y1 = torch.empty_like(y0)
    pkg.check(pkg.moe_forward(rc, c.xg, c.lg, c.layer.W, y1, None, ws))
    assert pkg.moe_get_status(ws) == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
