"""Runs the layer's reduced workloads through whichever build of the library
this process loads (MOE_GB300_LIB) and prints one JSON line: per workload the
device status after each call and a SHA-256 of every output's bytes.  Used by
tests/test_gpu_m_debug_build.py to compare the bounds-checked debug build
with the release build."""
import hashlib
import json
import os
import sys

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import moe_inputs as mi  # noqa: E402
from gpu_util import Case  # noqa: E402


def digest(*ts):
    h = hashlib.sha256()
    for t in ts:
        h.update(t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()[:16]


def main():
    import mixture_experts_layer_device_gb300 as pkg
    out = {"lib": pkg.LIB_PATH}
    for name in ("tiny", "qwen3.5-397b", "glm-5.2", "kimi-k2.7", "deepseek-v4-pro"):
        cfg = dict(mi.SMALL[name])
        c = Case(cfg, backward=cfg["backward"])
        L = c.layer
        y = L.forward(c.xg, c.lg, train=cfg["backward"]).clone()
        res = {"fwd_status": L.status(), "y": digest(y)}
        if cfg["backward"]:
            g = L.backward(c.dyg, c.xg)
            res["bwd_status"] = L.status()
            res["grads"] = digest(*[g[n] for n in sorted(g) if g[n] is not None])
        out[name] = res
    # the dispatch ring and NVFP4 experts
    cfg = dict(mi.SMALL["deepseek-v4-pro"])
    c = Case(cfg)
    rc = pkg.MoeConfig(c.layer.cfg.T, c.layer.cfg.d, c.layer.cfg.m, c.layer.cfg.E, c.layer.cfg.k, 0,
                       c.layer.cfg.dtype, 0, 256, 2)
    ws = torch.zeros(pkg.moe_workspace_bytes(rc), dtype=torch.uint8, device="cuda")
    y = torch.empty((cfg["T"], cfg["d"]), dtype=torch.bfloat16, device="cuda")
    pkg.check(pkg.moe_forward(rc, c.xg, c.lg, c.layer.W, y, None, ws))
    out["ring"] = {"fwd_status": pkg.moe_get_status(ws), "y": digest(y)}
    cfg = dict(mi.SMALL["deepseek-v4-pro"], m=512, fmt="nvfp4")
    c = Case(cfg)
    y = c.layer.forward(c.xg, c.lg).clone()
    out["nvfp4"] = {"fwd_status": c.layer.status(), "y": digest(y)}
    print(json.dumps(out))


if __name__ == "__main__":
    main()
