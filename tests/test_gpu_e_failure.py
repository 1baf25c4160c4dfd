"""Device-side failure detection without a GPU fault: a debug flag makes the
gate/up GEMM's load warp issue nothing, so the MMA warp's bounded wait runs out
(50 ms).  The call must come back, report MOE_ERR_TIMEOUT through
moe_get_status, and leave the CUDA context usable: the next normal call on the
same workspace gives the oracle's result."""
import time

import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import TOL, Case, rel

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "kimi-k2.7"])   # BF16 (CTA-pair GEMM) and MXFP8
def test_device_timeout_reported_and_context_survives(name):
    import mixture_experts_layer_device_gb300 as pkg
    cfg = dict(mi.SMALL[name])
    c = Case(cfg, backward=False)
    L = c.layer
    starve = pkg.MoeConfig(L.cfg.T, L.cfg.d, L.cfg.m, L.cfg.E, L.cfg.k, L.cfg.m_shared, L.cfg.dtype,
                           L.cfg.flags | pkg.MOE_FLAG_DEBUG_STARVE)
    y = torch.empty((cfg["T"], cfg["d"]), dtype=torch.bfloat16, device="cuda")
    t0 = time.time()
    pkg.check(pkg.moe_forward(starve, c.xg, c.lg, L.W, y, None, L.ws))
    assert pkg.moe_get_status(L.ws) == -6          # MOE_ERR_TIMEOUT
    assert time.time() - t0 < 30
    assert pkg.moe_get_status(L.ws) == 0           # reading clears the word
    y2 = L.forward(c.xg, c.lg)
    assert L.status() == 0
    y_ref, _ = c.oracle_forward()
    assert rel(mi.to_f64(y2), y_ref) < TOL[cfg["fmt"]]
