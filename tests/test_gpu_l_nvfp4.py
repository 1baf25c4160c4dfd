"""The NVFP4 variant of the expert GEMMs (forward): packed E2M1 operands with
an E4M3 scale per 16 along K and an fp32 second-level scale per tensor, on
tcgen05.mma kind::mxf4nvf4 (the pages say the method has no NVFP4 path --
"Mixture-of-Kittens" wiki page, Key claims, MXFP8 bullet -- so the format is
NVIDIA's published NVFP4, restated in oracle/nvfp4.py).

* weight preparation (moe_prepare_weights): codes, prepared scales and the
  experts' second-level scales bit-exact against the oracle's quantiser;
* dispatch: every routed row's codes and scales bit-exact (x's second-level
  scale from all T tokens);
* forward outputs within the MXFP8 tolerance of the oracle (codes of x and W
  are identical on both sides; what differs is the fp32 vs float64
  accumulation and the fp32 vs float64 h that the second quantiser sees),
  and bitwise reproducible;
* at the DeepSeek-V4-Pro shape, whole output rows of seeded tokens.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import TOL, Case, StreamedExperts, padded_rows, rel, unpack_tiled_scales
from oracle import moe as om
from oracle import numerics as nx
from oracle import nvfp4 as nv

pytestmark = pytest.mark.gpu

# reduced workloads with the structure of the DeepSeek-V4-Pro and Kimi-K2.7
# shapes (m a multiple of 256: NVFP4 stages are 256 deep along K)
NV_SMALL = {
    "deepseek-v4-pro": dict(T=1000, d=512, m=512, E=48, k=6, m_shared=0, fmt="nvfp4", bias="hot8", seed=14,
                            backward=False),
    "kimi-k2.7": dict(T=392, d=768, m=256, E=40, k=8, m_shared=256, fmt="nvfp4", bias="zipf", seed=13,
                      backward=False),
}


def _unpack_codes(t, rows, K):
    return nv.unpack_pairs(t.view(torch.uint8).reshape(rows, K // 2).cpu().numpy())


def test_weight_preparation_bit_exact():
    import mixture_experts_layer_device_gb300 as pkg
    rng = np.random.default_rng(7)
    E, d, m = 3, 512, 256
    w = rng.standard_normal((E, 2 * m, d)) / 20
    w[0, 5, :16] = 0.0                                              # an all-zero block
    w[1, 9, 40] = 3.0                                               # expert 1's amax, alone in its block
    w[2] *= 1e-3                                                    # a small-magnitude expert
    gu = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16)
    dn = torch.from_numpy((rng.standard_normal((E, d, m)) / 40).astype(np.float32)).to(torch.bfloat16)
    c = pkg.config(64, d, m, E, 2, 0, "nvfp4")
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device="cuda")
    out = dict(gu=u8(E * 2 * m * d // 2), gu_scale=u8(E * 2 * m * d // 16), dn=u8(E * d * m // 2),
               dn_scale=u8(E * d * m // 16), gu_gscale=torch.empty(E, device="cuda"),
               dn_gscale=torch.empty(E, device="cuda"))
    pkg.check(pkg.moe_prepare_weights(c, gu.cuda(), dn.cuda(), **out))
    torch.cuda.synchronize()
    for key, W, rows, K in (("gu", gu, 2 * m, d), ("dn", dn, d, m)):
        Wf = mi.to_f64(W)
        codes = _unpack_codes(out[key], E * rows, K)
        sf = unpack_tiled_scales(out[key + "_scale"].cpu().numpy(), E * rows, 2 * K)
        gs = out[key + "_gscale"].cpu().numpy()
        for e in range(E):
            s = nv.global_scale(np.abs(Wf[e]).max())
            assert gs[e] == s, key
            c_ref, s_ref = nv.nvfp4_quantize(Wf[e], s, axis=1)
            assert np.array_equal(codes[e * rows:(e + 1) * rows], c_ref), (key, e)
            assert np.array_equal(sf[e * rows:(e + 1) * rows, :K // 16], s_ref), (key, e)
    assert pkg.moe_prepare_weights(c, gu.cuda(), dn.cuda(), out["gu"], out["gu_scale"], out["dn"],
                                   out["dn_scale"]) == -1       # NVFP4 needs the second-level scales


@pytest.mark.parametrize("name", ["deepseek-v4-pro", "kimi-k2.7"])
def test_nvfp4_forward_matches_oracle(name):
    cfg = dict(NV_SMALL[name])
    c = Case(cfg, backward=False)
    L = c.layer
    y = L.forward(c.xg, c.lg).clone()
    assert L.status() == 0
    # dispatch: the routed rows' codes and scales, bit-exact
    counts, offsets, poff, inv = c.route_views(1)
    pr = padded_rows(counts, offsets, poff)
    d = cfg["d"]
    x = mi.to_f64(c.x)
    s_x = nv.global_scale(np.abs(x).max())
    assert L.view(1, "x_gscale", "f32", (1,)).item() == s_x
    c_ref, s_ref = nv.nvfp4_quantize(x[inv // cfg["k"]], s_x, axis=1)
    codes = nv.unpack_pairs(L.view(1, "xs", "u8", (L.Rp, d // 2)).cpu().numpy())
    sf = unpack_tiled_scales(c.buffer(1, "xs_sf"), L.Rp, 2 * d)
    assert np.array_equal(codes[pr], c_ref)
    assert np.array_equal(sf[pr, :d // 16], s_ref)
    # outputs
    y_ref, _ = c.oracle_forward()
    assert rel(mi.to_f64(y), y_ref) < TOL["mxfp8"]
    err = np.abs(mi.to_f64(y) - y_ref)
    assert err.max() <= 0.05 * np.abs(y_ref).max() + 1e-2
    # bitwise reproducible
    y2 = L.forward(c.xg, c.lg)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_nvfp4_rejects_training_and_unsupported_shapes():
    import mixture_experts_layer_device_gb300 as pkg
    assert pkg.moe_workspace_bytes(pkg.config(256, 512, 256, 8, 2, 0, "nvfp4", pkg.MOE_FLAG_BACKWARD)) == 0
    assert pkg.moe_workspace_bytes(pkg.config(256, 512, 384, 8, 2, 0, "nvfp4")) == 0        # m % 256
    assert pkg.moe_workspace_bytes(pkg.config(256, 512, 256, 8, 2, 0, "nvfp4", 0, 256)) == 0  # no ring


def test_full_size_nvfp4_forward_sampled_tokens():
    """DeepSeek-V4-Pro shape with NVFP4 experts: whole output rows of 32 seeded
    tokens (their experts' operands prepared by the oracle, streamed)."""
    from mixture_experts_layer_device_gb300.layer import MoELayer
    cfg = dict(mi.WORKLOADS["deepseek-v4-pro"], fmt="nvfp4")
    dev = torch.device("cuda")
    x, logits = mi.tokens(cfg, dev), mi.logits(cfg, dev)
    E, d, m = cfg["E"], cfg["d"], cfg["m"]
    gu_all = torch.empty((E, 2 * m, d), dtype=torch.bfloat16, device=dev)
    dn_all = torch.empty((E, d, m), dtype=torch.bfloat16, device=dev)
    for e in range(E):
        gu_all[e], dn_all[e] = mi.expert(cfg, e, dev)
    layer = MoELayer(cfg["T"], d, m, E, cfg["k"], "nvfp4", device=dev, stacked=(gu_all, dn_all))
    y = layer.forward(x, logits)
    assert layer.status() == 0
    tok = mi.sample_tokens(cfg, 32)
    lg = logits[tok].cpu().numpy()
    idx, _ = om.route(lg, cfg["k"])
    s_x = nv.global_scale(float(x.float().abs().max().item()))
    experts = StreamedExperts(cfg, gu_all, dn_all)
    try:
        experts.expect(np.unique(idx), forward=True, backward=False)
        y_ref, _ = om.forward(mi.to_f64(x[tok]), lg, experts, cfg["k"], "nvfp4", x_scale=s_x)
    finally:
        experts.close()
    y_gpu = mi.to_f64(y[tok])
    for i in range(len(tok)):
        assert rel(y_gpu[i], y_ref[i]) < TOL["mxfp8"], "token %d" % tok[i]
