"""Every fused MXFP8 quantisation point of the layer, byte for byte.

The pages fuse activation quantisation into the dispatch, the grouped GEMMs
and SwiGLU ("Mixture-of-Kittens" wiki page, Key claims, MXFP8 bullet; the
flowchart's "fused quantization").  Each point is checked by applying the
format's definition (the oracle's mx_quantize) to the exact values the kernel
quantised and comparing codes and scale bytes with what the kernel wrote:

* training dispatch: row codes (along d) and column-blocked codes x^T (blocks
  of 32 padded rows of one expert) of the bf16 token rows;
* gate/up epilogue: h codes (along m) from the fp32 SwiGLU output, and h^T
  codes from its bf16 rounding -- the fp32 h comes from the
  MOE_FLAG_DEBUG_DUMP hook;
* reverse combine (B1): dO = bf16(w * dy) with the fp32 product computed in
  NumPy float32 (IEEE, round to nearest even) from the GPU's own w, then row
  codes and column-blocked codes dO^T;
* SwiGLU-backward epilogue (B2): row and column-blocked codes of the bf16
  dG|dU values the dump hook stores.

The dumps are also compared with the oracle's own h and dGU (within the MXFP8
tolerance), so they are the layer's values and not some other buffer.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe as om
from oracle import numerics as nx

from gpu_util import Case, TOL, padded_rows, rel, unpack_tiled_scales

pytestmark = pytest.mark.gpu


def _u8(c, which, name, shape):
    return c.layer.view(which, name, "u8", shape).cpu().numpy()


def _check_rows(codes, sf_tiled, ref_vals, rows, K):
    """Row-blocked codes [rows, K] + tiled scales against mx_quantize(ref_vals, axis=1)."""
    c_ref, s_ref = nx.mx_quantize(ref_vals, axis=1)
    n = ref_vals.shape[0]
    assert np.array_equal(codes[:n], c_ref)
    assert np.array_equal(unpack_tiled_scales(sf_tiled, rows, K)[:n], s_ref)


def _check_cols(codesT, sfT_tiled, ref_vals, rows_T, Rp):
    """Column-blocked codes [C, Rp] (blocks of 32 padded rows) against
    mx_quantize(ref_vals^T, axis=1) over the written rows."""
    n = ref_vals.shape[0]
    c_ref, s_ref = nx.mx_quantize(np.ascontiguousarray(ref_vals.T), axis=1)
    assert np.array_equal(codesT[:, :n], c_ref)
    assert np.array_equal(unpack_tiled_scales(sfT_tiled, rows_T, Rp)[:, :n // 32], s_ref)


@pytest.mark.parametrize("name", ["kimi-k2.7", "deepseek-v4-pro"])
def test_fused_quantisation_points_bit_exact(name):
    import mixture_experts_layer_device_gb300 as pkg
    cfg = dict(mi.SMALL[name])
    c = Case(cfg, backward=True, flags=pkg.MOE_FLAG_DEBUG_DUMP)
    L = c.layer
    T, d, m, E, k = (cfg[n] for n in ("T", "d", "m", "E", "k"))
    Rp = L.Rp
    L.forward(c.xg, c.lg, train=True)
    L.backward(c.dyg, c.xg)
    assert L.status() == 0
    counts, offsets, poff, inv = c.route_views(0)
    pr = padded_rows(counts, offsets, poff)
    n = int(poff[E])                                   # rows written (whole padded experts)
    tok = np.full(n, -1)
    tok[pr] = inv // k
    slot = np.full(n, -1)
    slot[pr] = inv
    valid = tok >= 0

    # ---- training dispatch: x rows (exact bf16 values) in both orientations
    x = mi.to_f64(c.x)
    X = np.zeros((n, d))
    X[valid] = x[tok[valid]]
    _check_rows(_u8(c, 1, "xs", (Rp, d)), c.buffer(1, "xs_sf"), X, Rp, d)
    _check_cols(_u8(c, 0, "xT", (d, Rp)), c.buffer(0, "xT_sf"), X, d, Rp)

    # ---- gate/up epilogue: h codes from the fp32 SwiGLU output, h^T from its bf16 rounding
    h32 = L.view(1, "h_dump", "f32", (Rp, m))[:n].cpu().numpy().astype(np.float64)
    _check_rows(_u8(c, 1, "hq", (Rp, m)), c.buffer(1, "hq_sf"), h32, Rp, m)
    _check_cols(_u8(c, 0, "hT", (m, Rp)), c.buffer(0, "hT_sf"), nx.bf16_round(h32), m, Rp)
    y_ref, s = c.oracle_forward()
    assert rel(h32[pr], s["h"]) < TOL["mxfp8"]
    assert np.all(h32[~valid] == 0)

    # ---- B1: dO = bf16(fp32(w) * fp32(dy)) from the GPU's own combine weights
    w = L.view(0, "w", "f32", (T * k,)).cpu().numpy()
    dy32 = c.dy.float().numpy()
    dO = np.zeros((n, d))
    prod = w[slot[valid]][:, None].astype(np.float32) * dy32[tok[valid]]     # float32 IEEE multiply
    assert prod.dtype == np.float32
    dO[valid] = nx.bf16_round(prod.astype(np.float64))
    _check_rows(_u8(c, 1, "dOq", (Rp, d)), c.buffer(1, "dOq_sf"), dO, Rp, d)
    _check_cols(_u8(c, 1, "dOT", (d, Rp)), c.buffer(1, "dOT_sf"), dO, d, Rp)

    # ---- B2: dG|dU codes (row-blocked along 2m, and column-blocked) from the bf16 values
    dGU = L.view(1, "dGU_dump", "bf16", (Rp, 2 * m))[:n].float().cpu().numpy().astype(np.float64)
    _check_rows(_u8(c, 1, "dGUq", (Rp, 2 * m)), c.buffer(1, "dGUq_sf"), dGU, Rp, 2 * m)
    _check_cols(_u8(c, 1, "dGUT", (2 * m, Rp)), c.buffer(1, "dGUT_sf"), dGU, 2 * m, Rp)
    ref = om.backward(mi.to_f64(c.dy), x, c.oracle_experts(), k, "mxfp8", s, shared=c.oracle_shared(),
                      dw_experts=[])
    assert rel(dGU[pr], ref["dGU"]) < TOL["mxfp8"]
    assert np.all(dGU[~valid] == 0)


def test_dump_flag_changes_no_output():
    """The dump hook only adds stores: y, dx, dlogits and the weight gradients
    are bitwise those of the same layer without it."""
    import mixture_experts_layer_device_gb300 as pkg
    cfg = dict(mi.SMALL["kimi-k2.7"])
    outs = []
    for flags in (0, pkg.MOE_FLAG_DEBUG_DUMP):
        c = Case(cfg, backward=True, flags=flags)
        y = c.layer.forward(c.xg, c.lg, train=True).clone()
        g = c.layer.backward(c.dyg, c.xg)
        assert c.layer.status() == 0
        outs.append([y] + [g[n].clone() for n in ("dx", "dlogits", "dW_gu", "dW_dn", "dWs_gu", "dWs_dn")])
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
