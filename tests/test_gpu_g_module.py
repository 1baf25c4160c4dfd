"""The torch drop-in (autograd.Function + nn.Module) gives exactly what the C
ABI gives: y and every gradient (x, logits, the bf16 masters, the shared
expert) bitwise equal to direct moe_forward / moe_backward calls on the same
inputs, which the other GPU tests check against the oracle; an optimizer step
on the masters is seen by the next forward."""
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "kimi-k2.7"])   # BF16; MXFP8 + BF16 shared expert
def test_module_matches_direct_calls(name):
    from mixture_experts_layer_device_gb300.layer import MoELayer
    from mixture_experts_layer_device_gb300.module import MoE
    cfg = dict(mi.SMALL[name])
    T, d, m, E, k, ms = (cfg[n] for n in ("T", "d", "m", "E", "k", "m_shared"))
    dev = "cuda"
    gu, dn = (w.to(dev) for w in mi.experts(cfg))
    shared = mi.shared(cfg)
    shared = None if shared is None else tuple(w.to(dev) for w in shared)
    x, logits, dy = mi.tokens(cfg).to(dev), mi.logits(cfg).to(dev), mi.out_grad(cfg).to(dev)

    moe = MoE(T, d, m, E, k, cfg["fmt"], m_shared=ms, device=dev)
    with torch.no_grad():
        moe.W_gu.copy_(gu)
        moe.W_dn.copy_(dn)
        if shared is not None:
            moe.Ws_gu.copy_(shared[0])
            moe.Ws_dn.copy_(shared[1])
    xr, lr = x.clone().requires_grad_(True), logits.clone().requires_grad_(True)
    y = moe(xr, lr)
    (y.float() * dy.float()).sum().backward()

    ref = MoELayer(T, d, m, E, k, cfg["fmt"], shared=shared, backward=True, device=dev, stacked=(gu, dn))
    y_ref = ref.forward(x, logits, train=True)
    g = ref.backward(dy, x)
    assert torch.equal(y, y_ref)
    assert torch.equal(xr.grad, g["dx"])
    assert torch.equal(lr.grad, g["dlogits"])
    assert torch.equal(moe.W_gu.grad, g["dW_gu"])
    assert torch.equal(moe.W_dn.grad, g["dW_dn"])
    if shared is not None:
        assert torch.equal(moe.Ws_gu.grad, g["dWs_gu"])
        assert torch.equal(moe.Ws_dn.grad, g["dWs_dn"])


def test_module_sees_optimizer_steps_and_two_forwards():
    """Two forwards before their backwards keep separate activations, and the
    forward after an SGD step on the masters equals a fresh layer built from the
    updated masters."""
    from mixture_experts_layer_device_gb300.layer import MoELayer
    from mixture_experts_layer_device_gb300.module import MoE
    cfg = dict(mi.SMALL["kimi-k2.7"])
    T, d, m, E, k, ms = (cfg[n] for n in ("T", "d", "m", "E", "k", "m_shared"))
    dev = "cuda"
    torch.manual_seed(5)
    moe = MoE(T, d, m, E, k, cfg["fmt"], m_shared=ms, device=dev)
    x, logits = mi.tokens(cfg).to(dev), mi.logits(cfg).to(dev)
    x2 = (x.float() * 0.5).to(torch.bfloat16)
    dy = mi.out_grad(cfg).to(dev)
    # two forwards, then both backwards: each gradient matches its own forward
    y1 = moe(x, logits)
    y2 = moe(x2, logits)
    (y2.float() * dy.float()).sum().backward()
    g2 = moe.W_gu.grad.clone()
    moe.zero_grad()
    (y1.float() * dy.float()).sum().backward()
    g1 = moe.W_gu.grad.clone()
    shared = (moe.Ws_gu.detach(), moe.Ws_dn.detach())
    ref = MoELayer(T, d, m, E, k, cfg["fmt"], shared=shared, backward=True, device=dev,
                   stacked=(moe.W_gu.detach(), moe.W_dn.detach()))
    ref.forward(x, logits, train=True)
    assert torch.equal(ref.backward(dy, x)["dW_gu"], g1)
    ref.forward(x2, logits, train=True)
    assert torch.equal(ref.backward(dy, x2)["dW_gu"], g2)
    # an SGD step on the masters is used by the next forward
    with torch.no_grad():
        for p in moe.parameters():
            p.sub_(0.1 * p.grad)
    y3 = moe(x, logits)
    shared = (moe.Ws_gu.detach(), moe.Ws_dn.detach())
    fresh = MoELayer(T, d, m, E, k, cfg["fmt"], shared=shared, backward=True, device=dev,
                     stacked=(moe.W_gu.detach(), moe.W_dn.detach()))
    assert torch.equal(y3, fresh.forward(x, logits, train=True))
    assert not torch.equal(y3, y1)


def test_module_with_router_and_balance_term_matches_direct_calls():
    """router=True, aux_alpha > 0: the fused function's outputs and gradients
    equal the chain router_forward -> forward -> backward -> router_backward,
    and the load-balancing loss is exposed."""
    from mixture_experts_layer_device_gb300.layer import MoELayer
    from mixture_experts_layer_device_gb300.module import MoE
    cfg = dict(mi.SMALL["kimi-k2.7"])
    T, d, m, E, k, ms = (cfg[n] for n in ("T", "d", "m", "E", "k", "m_shared"))
    dev, alpha = "cuda", 0.01
    torch.manual_seed(9)
    moe = MoE(T, d, m, E, k, cfg["fmt"], m_shared=ms, device=dev, router=True, aux_alpha=alpha)
    x, dy = mi.tokens(cfg).to(dev), mi.out_grad(cfg).to(dev)
    xr = x.clone().requires_grad_(True)
    y = moe(xr)
    aux = float(moe.aux_loss())
    (y.float() * dy.float()).sum().backward()

    shared = (moe.Ws_gu.detach(), moe.Ws_dn.detach())
    ref = MoELayer(T, d, m, E, k, cfg["fmt"], shared=shared, backward=True, device=dev,
                   stacked=(moe.W_gu.detach(), moe.W_dn.detach()), aux_alpha=alpha)
    W_r = moe.W_r.detach()
    logits = ref.router_logits(x, W_r)
    y_ref = ref.forward(x, logits, train=True)
    aux_ref = float(ref.view(1, "aux", "f32", (1,))[0])
    g = ref.backward(dy, x)
    dW_r = torch.empty_like(W_r)
    ref.router_backward(g["dlogits"], x, W_r, g["dx"], dW_r)
    assert torch.equal(y, y_ref)
    assert aux == aux_ref and aux > 0
    assert torch.equal(xr.grad, g["dx"])
    assert torch.equal(moe.W_r.grad, dW_r)
    assert torch.equal(moe.W_gu.grad, g["dW_gu"])
    assert torch.equal(moe.W_dn.grad, g["dW_dn"])
    assert torch.equal(moe.Ws_gu.grad, g["dWs_gu"])
