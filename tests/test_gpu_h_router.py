"""GPU parity of the router projection and of the load-balancing term against
the oracle (oracle/router.py).

Tolerances: the loss, P and the gradient rows are fp32 softmax arithmetic
(expf, one division, fixed-order sums of at most T*E terms), so relative
errors stay near 1e-6; 1e-5 is used.  The router logits are an fp32-accumulated
bf16 GEMM over d: relative Frobenius error 1e-5.  The router backward's
outputs are rounded to bf16, so they are compared within the BF16 tolerance
of the layer (5e-3)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import TOL, rel
from oracle import moe as om
from oracle import router as orr

pytestmark = pytest.mark.gpu


def _layer(cfg, alpha):
    import mixture_experts_layer_device_gb300 as pkg
    from mixture_experts_layer_device_gb300.layer import MoELayer
    gu, dn = (w.cuda() for w in mi.experts(cfg))
    shared = mi.shared(cfg)
    shared = None if shared is None else tuple(w.cuda() for w in shared)
    L = MoELayer(cfg["T"], cfg["d"], cfg["m"], cfg["E"], cfg["k"], cfg["fmt"], shared=shared, backward=True,
                 device="cuda", stacked=(gu, dn))
    c = L.cfg
    L.cfg = pkg.MoeConfig(c.T, c.d, c.m, c.E, c.k, c.m_shared, c.dtype, c.flags, 0, 0, alpha)
    L.ws = torch.zeros(pkg.moe_workspace_bytes(L.cfg), dtype=torch.uint8, device="cuda")
    L.saved = torch.zeros(pkg.moe_saved_bytes(L.cfg), dtype=torch.uint8, device="cuda")
    return L


@pytest.mark.parametrize("name", ["tiny", "kimi-k2.7", "deepseek-v4-pro"])
def test_balance_loss_and_gradient_match_oracle(name):
    cfg = dict(mi.SMALL[name])
    alpha = 0.01
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    L = _layer(cfg, alpha)
    x, logits, dy = mi.tokens(cfg).cuda(), mi.logits(cfg).cuda(), mi.out_grad(cfg).cuda()
    L.forward(x, logits, train=True)
    assert L.status() == 0
    aux = L.view(1, "aux", "f32", (1 + 2 * E,)).cpu().numpy().astype(np.float64)
    counts = L.view(0, "counts", "i32", (E,)).cpu().numpy()
    lg = logits.cpu().numpy()
    loss, grad = orr.aux_loss(lg, counts, k, alpha)
    f, P, _ = orr.balance_terms(lg, counts, k)
    assert abs(aux[0] - loss) <= 1e-5 * abs(loss)
    assert rel(aux[1:1 + E], P) < 1e-5
    assert rel(aux[1 + E:], f) < 1e-6
    g_aux = L.view(0, "aux_grad", "f32", (T, E)).cpu().numpy().astype(np.float64)
    assert rel(g_aux, grad) < 1e-5
    # the backward adds it to dlogits: compare with the same layer without the term
    g1 = L.backward(dy, x)
    dl_with = g1["dlogits"].cpu().numpy().astype(np.float64)
    L0 = _layer(cfg, 0.0)
    L0.forward(x, logits, train=True)
    dl_without = L0.backward(dy, x)["dlogits"].cpu().numpy().astype(np.float64)
    assert np.abs((dl_with - dl_without) - grad).max() < 1e-6 * max(1.0, np.abs(grad).max()) + 1e-7
    # bitwise reproducible
    L.forward(x, logits, train=True)
    aux2 = L.view(1, "aux", "f32", (1 + 2 * E,)).cpu().numpy()
    assert np.array_equal(aux2, aux.astype(np.float32))


def test_router_forward_and_backward_match_oracle():
    import mixture_experts_layer_device_gb300 as pkg
    cfg = dict(mi.SMALL["kimi-k2.7"])
    T, d, E = cfg["T"], cfg["d"], cfg["E"]
    g = torch.Generator().manual_seed(77)
    x = mi.tokens(cfg).cuda()
    W_r = (torch.randn((E, d), generator=g) * d ** -0.5).to(torch.bfloat16).cuda()
    c = pkg.config(T, d, cfg["m"], E, cfg["k"], cfg["m_shared"], cfg["fmt"], pkg.MOE_FLAG_BACKWARD)
    ws = torch.zeros(pkg.moe_workspace_bytes(c), dtype=torch.uint8, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    pkg.check(pkg.moe_router_forward(c, x, W_r, logits, ws))
    torch.cuda.synchronize()
    ref = orr.router_logits(mi.to_f64(x), mi.to_f64(W_r))
    assert rel(logits.cpu().numpy(), ref) < 1e-5
    # backward: dx updated in place (checked from zero, then on top of a layer's
    # dx, where one bf16 rounding of the sum hides increments below its spacing)
    dlog = (torch.randn((T, E), generator=g) * 1e-2).cuda()
    dW = torch.empty((E, d), dtype=torch.bfloat16, device="cuda")
    for dx0 in (torch.zeros((T, d), dtype=torch.bfloat16, device="cuda"), mi.out_grad(cfg).cuda()):
        dx = dx0.clone()
        pkg.check(pkg.moe_router_backward(c, dlog, x, W_r, dx, dW, ws))
        torch.cuda.synchronize()
        dx_ref, dW_ref = orr.router_backward(dlog.cpu().numpy().astype(np.float64), mi.to_f64(x),
                                             mi.to_f64(W_r), mi.to_f64(dx0))
        assert rel(mi.to_f64(dx), dx_ref) < TOL["bf16"]
        assert rel(mi.to_f64(dW), dW_ref) < TOL["bf16"]
    # the logits feed the layer: route on them like any other logits
    idx, _ = om.route(logits.cpu().numpy(), cfg["k"])
    assert idx.shape == (T, cfg["k"])
