"""The forward + backward step is capturable into a CUDA graph: every library
call is stream-ordered on the caller's stream, with no host synchronisation,
and one-time launch-configuration queries are memoised before the capture.
Replays give bitwise the results of eager calls, for the inputs captured with
and for new inputs copied into the same buffers."""
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu


def _layer(cfg, ring_rows=0):
    from mixture_experts_layer_device_gb300.layer import MoELayer
    gu, dn = (w.cuda() for w in mi.experts(cfg))
    shared = mi.shared(cfg)
    shared = None if shared is None else tuple(w.cuda() for w in shared)
    return MoELayer(cfg["T"], cfg["d"], cfg["m"], cfg["E"], cfg["k"], cfg["fmt"], shared=shared, backward=True,
                    device="cuda", stacked=(gu, dn), ring_rows=ring_rows)


def _eager(L, x, logits, dy):
    y = L.forward(x, logits, train=True).clone()
    g = L.backward(dy, x)
    assert L.status() == 0
    return y, {k: (None if v is None else v.clone()) for k, v in g.items()}


@pytest.mark.parametrize("name,ring_rows", [("tiny", 0), ("kimi-k2.7", 0), ("kimi-k2.7", 256)])
def test_graph_replay_matches_eager(name, ring_rows):
    cfg = dict(mi.SMALL[name]) if name != "tiny" else dict(mi.WORKLOADS["tiny"])
    L = _layer(cfg, ring_rows)
    x, logits, dy = mi.tokens(cfg).cuda(), mi.logits(cfg).cuda(), mi.out_grad(cfg).cuda()
    y_ref, g_ref = _eager(L, x, logits, dy)

    y = torch.empty_like(y_ref)
    grads = L.alloc_grads()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):               # warm-up on a side stream, as capture requires
        L.forward(x, logits, y=y, train=True, stream=side)
        L.backward(dy, x, grads=grads, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        st = torch.cuda.current_stream()
        L.forward(x, logits, y=y, train=True, stream=st)
        L.backward(dy, x, grads=grads, stream=st)
    y.zero_()
    for v in grads.values():
        if v is not None:
            v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert L.status() == 0
    assert torch.equal(y, y_ref)
    for n, v in g_ref.items():
        if v is not None:
            assert torch.equal(grads[n], v), n
    # new inputs in the captured buffers
    g = torch.Generator().manual_seed(123)
    x2 = (torch.randn(x.shape, generator=g)).to(torch.bfloat16).cuda()
    l2 = torch.randn(logits.shape, generator=g).cuda()
    y2_ref, g2_ref = _eager(L, x2, l2, dy)
    x.copy_(x2)
    logits.copy_(l2)
    graph.replay()
    torch.cuda.synchronize()
    assert L.status() == 0
    assert torch.equal(y, y2_ref)
    for n, v in g2_ref.items():
        if v is not None:
            assert torch.equal(grads[n], v), n
