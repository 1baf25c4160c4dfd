"""Parity at the full workload sizes, in the launch configuration bench.py
times (stacked weight preparation, one moe_forward / moe_backward over all T
tokens), on outputs the oracle can compute one by one:

* whole output rows of 256 seeded tokens per workload (all their experts and
  the shared expert);
* on the Kimi-K2.7 fwd+bwd step, dx and dlogits rows of the same 256 tokens,
  and the weight gradients of 4 seeded experts over all their rows, one of
  them the most loaded expert (its wgrad reduces about 16 k rows);
* every gradient element written, and all-zero dW for experts without rows.

The oracle's weight operands are prepared expert by expert by a worker pool
(StreamedExperts), so host memory holds a few experts' operands at a time."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import TOL, StreamedExperts, rel
from oracle import moe as om

pytestmark = pytest.mark.gpu

N_TOK = 256


def build(name, backward):
    from mixture_experts_layer_device_gb300.layer import MoELayer
    cfg = dict(mi.WORKLOADS[name])
    dev = torch.device("cuda")
    x, logits = mi.tokens(cfg, dev), mi.logits(cfg, dev)
    E, d, m = cfg["E"], cfg["d"], cfg["m"]
    gu_all = torch.empty((E, 2 * m, d), dtype=torch.bfloat16, device=dev)
    dn_all = torch.empty((E, d, m), dtype=torch.bfloat16, device=dev)
    for e in range(E):
        gu_all[e], dn_all[e] = mi.expert(cfg, e, dev)
    shared = mi.shared(cfg, dev)
    layer = MoELayer(cfg["T"], d, m, E, cfg["k"], cfg["fmt"], shared=shared, backward=backward, device=dev,
                     stacked=(gu_all, dn_all))
    return cfg, x, logits, gu_all, dn_all, shared, layer


def check_rows(got, ref, tok, tol, what):
    for i in range(len(tok)):
        assert rel(got[i], ref[i]) < tol, "%s of token %d" % (what, tok[i])


@pytest.mark.parametrize("name", ["qwen3.5-397b", "glm-5.2", "deepseek-v4-pro"])
def test_full_size_forward_sampled_tokens(name):
    cfg, x, logits, gu_all, dn_all, shared, layer = build(name, backward=False)
    y = layer.forward(x, logits)
    assert layer.status() == 0
    tok = mi.sample_tokens(cfg, N_TOK)
    lg = logits[tok].cpu().numpy()
    idx, _ = om.route(lg, cfg["k"])
    sh = None if shared is None else tuple(mi.to_f64(w) for w in shared)
    experts = StreamedExperts(cfg, gu_all, dn_all)
    try:
        experts.expect(np.unique(idx), forward=True, backward=False)
        y_ref, _ = om.forward(mi.to_f64(x[tok]), lg, experts, cfg["k"], cfg["fmt"], shared=sh)
    finally:
        experts.close()
    check_rows(mi.to_f64(y[tok]), y_ref, tok, TOL[cfg["fmt"]], "y")


def test_full_size_forward_backward_sampled():
    """Kimi-K2.7 shape, MXFP8 + BF16 shared expert, the step bench.py times."""
    cfg, x, logits, gu_all, dn_all, shared, layer = build("kimi-k2.7", backward=True)
    dy = mi.out_grad(cfg, x.device)
    y_inf = layer.forward(x, logits).clone()
    y = layer.forward(x, logits, train=True)
    assert torch.equal(y_inf.view(torch.int16), y.view(torch.int16))    # inference == training forward
    grads = layer.alloc_grads()
    for v in grads.values():
        if v is not None:
            v.fill_(float("nan"))  # every element must be written by the backward
    g = layer.backward(dy, x, grads=grads)
    assert layer.status() == 0
    k, fmt, tol = cfg["k"], cfg["fmt"], TOL[cfg["fmt"]]
    tok = mi.sample_tokens(cfg, N_TOK)
    lg = logits[tok].cpu().numpy()
    idx, _ = om.route(lg, k)
    counts = layer.view(0, "counts", "i32", (cfg["E"],)).cpu().numpy()
    hot = int(np.argmax(counts))
    others = mi.sample_experts(np.where(np.arange(cfg["E"]) == hot, 0, counts), cfg["seed"], n=3)
    e_dws = sorted([hot] + [int(e) for e in others])
    assert len(set(e_dws)) == 4 and counts[hot] > 8192
    sh = None if shared is None else tuple(mi.to_f64(w) for w in shared)
    xs, dys = mi.to_f64(x[tok]), mi.to_f64(dy[tok])
    need = np.unique(idx)
    experts = StreamedExperts(cfg, gu_all, dn_all)
    try:
        experts.expect(need, forward=True, backward=False)
        y_ref, saved = om.forward(xs, lg, experts, k, fmt, shared=sh)
        experts.expect(need, forward=False, backward=True)
        ref = om.backward(dys, xs, experts, k, fmt, saved, shared=sh, dw_experts=[])
        check_rows(mi.to_f64(y[tok]), y_ref, tok, tol, "y")
        check_rows(mi.to_f64(g["dx"][tok]), ref["dx"], tok, tol, "dx")
        check_rows(g["dlogits"][tok].cpu().numpy().astype(np.float64), ref["dlogits"], tok, tol, "dlogits")
        # dW of each sampled expert: every row routed to it, in the schedule's (slot) order
        idx_all = layer.view(0, "idx", "i32", (cfg["T"], k)).cpu().numpy()
        w_all = layer.view(0, "w", "f32", (cfg["T"], k)).cpu().numpy().astype(np.float64)
        experts.expect(e_dws, forward=True, backward=True)
        for e_dw in e_dws:
            slots = np.nonzero(idx_all.reshape(-1) == e_dw)[0]
            assert slots.size == counts[e_dw] > 0
            toks = torch.as_tensor(slots // k, device=x.device)
            W_gu, W_dn, ops = experts[e_dw]
            X = mi.to_f64(x[toks])
            fw = om.expert_forward(X, W_gu, W_dn, fmt, ops)
            dO = om._rnd(fmt)(w_all.reshape(-1)[slots][:, None] * mi.to_f64(dy[toks]))
            bw = om.expert_backward(dO, X, fw["GU_saved"], fw["h_saved"], W_gu, W_dn, fmt, ops)
            assert rel(mi.to_f64(g["dW_gu"][e_dw]), bw["dW_gu"]) < tol, "dW_gu of expert %d" % e_dw
            assert rel(mi.to_f64(g["dW_dn"][e_dw]), bw["dW_dn"]) < tol, "dW_dn of expert %d" % e_dw
            del fw, bw, X, dO
    finally:
        experts.close()
    # every dW element is written, and an expert that received no rows has an
    # all-zero gradient (the Zipf-biased router leaves many experts empty)
    empty = torch.as_tensor(counts == 0, device=x.device)
    assert bool(empty.any())
    for name in ("dW_gu", "dW_dn"):
        for e0 in range(0, cfg["E"], 32):
            blk = g[name][e0:e0 + 32]
            assert not bool(torch.isnan(blk).any()), "%s: unwritten elements near expert %d" % (name, e0)
            z = empty[e0:e0 + 32]
            if bool(z.any()):
                assert not bool(blk[z].any()), "%s of an empty expert near %d" % (name, e0)
    for name in ("dx", "dlogits", "dWs_gu", "dWs_dn"):
        assert not bool(torch.isnan(g[name]).any()), name


def test_full_size_ring_bitwise_equal():
    """DeepSeek-V4-Pro shape through an 8,192-row ring (64 slots, 8 gather SMs),
    well below the rows of each hot expert: the whole output equals the
    materialised dispatch's bit for bit, from a much smaller workspace."""
    import mixture_experts_layer_device_gb300 as pkg
    cfg, x, logits, gu_all, dn_all, shared, layer = build("deepseek-v4-pro", backward=False)
    y0 = layer.forward(x, logits)
    assert layer.status() == 0
    counts = layer.view(1, "counts", "i32", (cfg["E"],)).cpu().numpy()
    assert counts.max() > 8192
    c = layer.cfg
    rc = pkg.MoeConfig(c.T, c.d, c.m, c.E, c.k, c.m_shared, c.dtype, c.flags, 8192, 8)
    ws = torch.empty(pkg.moe_workspace_bytes(rc), dtype=torch.uint8, device=x.device)
    assert ws.numel() < layer.ws.numel()
    y1 = torch.empty_like(y0)
    pkg.check(pkg.moe_forward(rc, x, logits, layer.W, y1, None, ws))
    assert pkg.moe_get_status(ws) == 0
    assert torch.equal(y0, y1)
