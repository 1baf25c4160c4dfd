"""GPU parity of the backward pass against the oracle (reduced-size workloads),
and bitwise determinism of the gradients."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import TOL, Case, rel
from oracle import moe as om

pytestmark = pytest.mark.gpu


def run(case):
    case.layer.forward(case.xg, case.lg, train=True)
    grads = case.layer.alloc_grads()
    for v in grads.values():
        if v is not None:
            v.fill_(float("nan"))  # every element must be written by the backward
    g = case.layer.backward(case.dyg, case.xg, grads=grads)
    assert case.layer.status() == 0
    return g


@pytest.mark.parametrize("name", ["tiny", "kimi-k2.7", "qwen3.5-397b", "deepseek-v4-pro"])
def test_backward_matches_oracle(name):
    cfg = dict(mi.SMALL[name])
    c = Case(cfg, backward=True)
    g = run(c)
    y_ref, saved = c.oracle_forward()
    ref = om.backward(mi.to_f64(c.dy), mi.to_f64(c.x), c.oracle_experts(), cfg["k"], cfg["fmt"], saved,
                      shared=c.oracle_shared())
    tol = TOL[cfg["fmt"]]
    assert rel(g["dx"].float().cpu().numpy(), ref["dx"]) < tol, "dx"
    assert rel(g["dlogits"].cpu().numpy(), ref["dlogits"]) < tol, "dlogits"
    mask = np.zeros((cfg["T"], cfg["E"]), bool)
    np.put_along_axis(mask, saved["idx"], True, 1)
    assert np.all(g["dlogits"].cpu().numpy()[~mask] == 0)
    dW_gu = g["dW_gu"].float().cpu().numpy()
    dW_dn = g["dW_dn"].float().cpu().numpy()
    for e in range(cfg["E"]):
        if saved["counts"][e] == 0:
            assert np.all(dW_gu[e] == 0) and np.all(dW_dn[e] == 0), "empty expert %d" % e
        else:
            assert rel(dW_gu[e], ref["dW_gu"][e]) < tol, "dW_gu[%d]" % e
            assert rel(dW_dn[e], ref["dW_dn"][e]) < tol, "dW_dn[%d]" % e
    if cfg["m_shared"]:
        assert rel(g["dWs_gu"].float().cpu().numpy(), ref["dWs_gu"]) < tol
        assert rel(g["dWs_dn"].float().cpu().numpy(), ref["dWs_dn"]) < tol


def test_backward_bitwise_deterministic():
    c = Case(dict(mi.SMALL["kimi-k2.7"]), backward=True)
    g1 = {k: (v.clone() if v is not None else None) for k, v in run(c).items()}
    g2 = run(c)
    for k in g1:
        if g1[k] is not None:
            a, b = g1[k], g2[k]
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b), k
