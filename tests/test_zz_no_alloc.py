"""moe_route_noalloc: routing for callers that cannot call cudaMalloc (for
example code running under a framework that owns all device memory through its
own arena).  It must give exactly what moe_route gives, call after call, while
using only the library's fixed device scratch array.  Collected last so that a
run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import mixture_experts_layer_device_gb300 as m
    return m


def _outputs(T, E, k):
    dev = "cuda"
    return (torch.empty((T, k), dtype=torch.int32, device=dev), torch.empty((T, k), dtype=torch.float32, device=dev),
            torch.empty(E, dtype=torch.int32, device=dev), torch.empty(E + 1, dtype=torch.int32, device=dev),
            torch.empty(T * k, dtype=torch.int32, device=dev))


def _route_ws(pkg, cfg, logits):
    ws = torch.empty(pkg.moe_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    out = _outputs(cfg.T, cfg.E, cfg.k)
    pkg.check(pkg.moe_route(cfg, logits, *out, ws))
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out]


def _route_noalloc(pkg, cfg, logits):
    out = _outputs(cfg.T, cfg.E, cfg.k)
    pkg.check(pkg.moe_route_noalloc(cfg, logits, *out))
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out]


def test_noalloc_route_matches_route_on_consecutive_calls(pkg):
    shapes = [(16384, 384, 8, 3.0), (1000, 37, 5, 0.0), (32768, 384, 6, 0.0)]   # last: the largest workload
    for i, (T, E, k, skew) in enumerate(shapes):
        g = torch.Generator().manual_seed(100 + i)
        logits = torch.randn((T, E), generator=g)
        logits[:, : max(1, E // 16)] += skew
        logits = logits.cuda()
        cfg = pkg.config(T, 256, 128, E, k)
        ref = _route_ws(pkg, cfg, logits)
        for _ in range(2):                      # two calls in a row share the scratch array
            got = _route_noalloc(pkg, cfg, logits)
            for name, a, b in zip(("idx", "w", "counts", "offsets", "perm"), got, ref):
                assert np.array_equal(a, b), name     # same kernels, same bits (w included)


def test_noalloc_route_rejects_oversized_shapes(pkg):
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    big = pkg.config(pkg_max_slots() // 8 + 1, 256, 128, 64, 8)
    assert pkg.moe_route_noalloc(big, dummy, dummy, dummy, dummy, dummy, dummy) == -2
    many = pkg.config(64, 256, 128, 2048, 8)
    assert pkg.moe_route_noalloc(many, dummy, dummy, dummy, dummy, dummy, dummy) == -2
    assert pkg.moe_route_noalloc(pkg.config(64, 256, 128, 16, 2), None, dummy, dummy, dummy, dummy, dummy) == -1


def pkg_max_slots():
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")).read()
    return int(re.search(r"#define MOE_ROUTE_NOALLOC_MAX_SLOTS (\d+)", hdr).group(1))
