"""Degenerate and ragged layer shapes, forward and backward, against the
oracle, in both expert formats: one token (most experts empty), every expert
selected (k = E), every token on the same two experts (one expert spans
several 128-row tiles, all others are empty: the wgrads write all-zero tiles),
ragged token counts, and a thousand experts (a large grouped-GEMM schedule,
most experts with zero to two rows).  Gradients are prefilled with NaN so
that an element the backward never writes fails the comparison."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import TOL, Case, rel
from oracle import moe as om

pytestmark = pytest.mark.gpu

SHAPES = {
    "one-token": dict(T=1, d=256, m=128, E=8, k=2),
    "k-equals-E": dict(T=37, d=256, m=128, E=5, k=5),
    "all-on-two": dict(T=300, d=256, m=128, E=16, k=2, skew=True),
    "ragged": dict(T=129, d=512, m=256, E=12, k=3),
    "many-experts": dict(T=200, d=256, m=128, E=1000, k=4),
}


def _case(shape, fmt):
    cfg = dict(SHAPES[shape])
    skew = cfg.pop("skew", False)
    cfg.update(m_shared=0, fmt=fmt, bias="none", seed=31, backward=True)
    c = Case(cfg, backward=True)
    if skew:  # experts 0 and 1 win every token by a wide margin
        c.logits = c.logits.clone()
        c.logits[:, :2] += 50.0
        c.lg = c.logits.cuda()
    return cfg, c


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_edge_shapes_forward_backward(shape, fmt):
    cfg, c = _case(shape, fmt)
    L = c.layer
    y = L.forward(c.xg, c.lg, train=True)
    grads = L.alloc_grads()
    for v in grads.values():
        if v is not None:
            v.fill_(float("nan"))
    g = L.backward(c.dyg, c.xg, grads=grads)
    assert L.status() == 0
    y_ref, saved = c.oracle_forward()
    ref = om.backward(mi.to_f64(c.dy), mi.to_f64(c.x), c.oracle_experts(), cfg["k"], fmt, saved)
    tol = TOL[fmt]
    assert rel(mi.to_f64(y), y_ref) < tol, "y"
    assert rel(mi.to_f64(g["dx"]), ref["dx"]) < tol, "dx"
    dl = g["dlogits"].cpu().numpy().astype(np.float64)
    assert not np.isnan(dl).any()
    assert rel(dl, ref["dlogits"]) < tol, "dlogits"
    dW_gu = g["dW_gu"].float().cpu().numpy()
    dW_dn = g["dW_dn"].float().cpu().numpy()
    assert not np.isnan(dW_gu).any() and not np.isnan(dW_dn).any()
    for e in range(cfg["E"]):
        if saved["counts"][e] == 0:
            assert np.all(dW_gu[e] == 0) and np.all(dW_dn[e] == 0), "empty expert %d" % e
        else:
            assert rel(dW_gu[e], ref["dW_gu"][e]) < tol, "dW_gu[%d]" % e
            assert rel(dW_dn[e], ref["dW_dn"][e]) < tol, "dW_dn[%d]" % e
    if shape == "all-on-two":
        assert list(np.nonzero(saved["counts"])[0]) == [0, 1]
        assert saved["counts"][0] == cfg["T"] > 256  # several 128-row tiles of one expert
