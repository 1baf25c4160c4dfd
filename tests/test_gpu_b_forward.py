"""GPU parity of the forward pass against the oracle, element by element, on
reduced-size workloads with the structure of each named workload (several GEMM
tiles, ragged tails, skewed loads, empty experts), plus the dispatch
quantisation bit-exact and run-to-run bitwise determinism."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import TOL, Case, padded_rows, rel, unpack_tiled_scales
from oracle import moe as om
from oracle import numerics as nx

pytestmark = pytest.mark.gpu


def small(name, **over):
    c = dict(mi.SMALL[name])
    c.update(over)
    return c


def run_forward(case, train=True):
    y = case.layer.forward(case.xg, case.lg, train=train)
    assert case.layer.status() == 0
    return y


def saved_rows(case, name, width, dtype="bf16"):
    """Rows [0, poff[E]) of a saved row buffer (the rows past the last expert's
    padded block are never written)."""
    L = case.layer
    n = int(L.view(0, "poff", "i32", (L.E + 1,))[L.E].item())
    t = L.view(0, name, dtype, (L.Rp, width))[:n]
    return t.float().cpu().numpy().astype(np.float64)


def check_saved_h(case, s, pr, tol):
    """The h a training forward keeps for the backward: bf16 rows (BF16), or
    for MXFP8 the column-blocked codes h^T [m, Rp] (blocks of 32 padded rows
    of one expert), compared after decoding with the oracle's column-blocked
    MX round trip of its own h, expert by expert."""
    cfg, L = case.cfg, case.layer
    m = cfg["m"]
    if cfg["fmt"] == "bf16":
        assert rel(saved_rows(case, "h", m)[pr], s["h"]) < tol
        return
    codes = L.view(0, "hT", "u8", (m, L.Rp)).cpu().numpy()
    sf = unpack_tiled_scales(case.buffer(0, "hT_sf"), m, L.Rp)
    h_gpu = nx.mx_dequantize(codes, sf, axis=1).T                  # [Rp, m]
    ref = np.zeros_like(s["h"])
    offs = s["offsets"]
    for e in range(cfg["E"]):
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if r1 > r0:
            ref[r0:r1] = om._col_blocks(s["h"][r0:r1])
    assert rel(h_gpu[pr], ref) < tol


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_single_expert_ffn(fmt):
    """E = 1, k = 1: the layer is one SwiGLU FFN; checks GEMM1, SwiGLU and GEMM2 alone."""
    cfg = dict(T=200, d=256, m=128, E=1, k=1, m_shared=0, fmt=fmt, bias="none", seed=21, backward=False)
    c = Case(cfg, backward=True)
    y = run_forward(c).float().cpu().numpy()
    y_ref, s = c.oracle_forward()
    counts, offsets, poff, _ = c.route_views(0)
    assert list(poff) == [0, 256]
    pr = padded_rows(counts, offsets, poff)
    assert rel(saved_rows(c, "GU", 2 * cfg["m"])[pr], s["GU"]) < TOL[fmt] / 5, "gate/up GEMM"
    check_saved_h(c, s, pr, TOL[fmt])
    assert rel(saved_rows(c, "o", cfg["d"])[pr], s["o"]) < TOL[fmt], "down GEMM"
    assert rel(y, y_ref) < TOL[fmt]


@pytest.mark.parametrize("name", mi.ORDER)
def test_forward_matches_oracle(name):
    cfg = small(name)
    c = Case(cfg, backward=True)
    y = run_forward(c).float().cpu().numpy()
    y_ref, s = c.oracle_forward()
    counts, offsets, poff, _ = c.route_views(0)
    assert np.array_equal(counts, s["counts"]) and np.array_equal(offsets, s["offsets"])
    assert np.array_equal(poff[1:] - poff[:-1], (counts + 127) // 128 * 128)
    pr = padded_rows(counts, offsets, poff)
    tol = TOL[cfg["fmt"]]
    assert rel(saved_rows(c, "GU", 2 * cfg["m"])[pr], s["GU"]) < tol
    check_saved_h(c, s, pr, tol)
    assert rel(saved_rows(c, "o", cfg["d"])[pr], s["o"]) < tol
    assert rel(y, y_ref) < tol
    # elementwise: no single output is far off (catches a wrong row or block)
    err = np.abs(y - y_ref)
    assert err.max() <= 0.05 * np.abs(y_ref).max() + 1e-2


@pytest.mark.parametrize("name", ["glm-5.2", "deepseek-v4-pro"])
def test_dispatch_quantisation_bit_exact(name):
    cfg = small(name)
    c = Case(cfg, backward=False)
    run_forward(c, train=False)
    L = c.layer
    counts, offsets, poff, inv = c.route_views(1)
    pr = padded_rows(counts, offsets, poff)
    d = cfg["d"]
    codes = L.view(1, "xs", "u8", (L.Rp, d)).cpu().numpy()
    sf = c.buffer(1, "xs_sf")
    x = mi.to_f64(c.x)
    c_ref, s_ref = nx.mx_quantize(x[inv // cfg["k"]], axis=1)
    assert np.array_equal(codes[pr], c_ref)
    assert np.array_equal(unpack_tiled_scales(sf, L.Rp, d)[pr], s_ref)
    # padding rows are zero codes with scale byte 0
    pad = np.setdiff1d(np.arange(int(poff[-1])), pr)
    assert np.all(codes[pad] == 0) and np.all(unpack_tiled_scales(sf, L.Rp, d)[pad] == 0)


@pytest.mark.parametrize("name", ["qwen3.5-397b", "kimi-k2.7"])
def test_forward_bitwise_deterministic(name):
    cfg = small(name)
    c = Case(cfg, backward=True)
    y1 = run_forward(c).clone()
    o1 = c.layer.view(0, "o", "bf16", (c.layer.Rp, cfg["d"])).clone()
    y2 = run_forward(c, train=False)
    y3 = run_forward(c)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    counts, offsets, poff, _ = c.route_views(0)
    pr = torch.as_tensor(padded_rows(counts, offsets, poff), device="cuda")
    o3 = c.layer.view(0, "o", "bf16", (c.layer.Rp, cfg["d"]))
    assert torch.equal(o1[pr].view(torch.int16), o3[pr].view(torch.int16))


@pytest.mark.parametrize("name", ["kimi-k2.7", "deepseek-v4-pro"])
def test_tile_order_is_a_token_sorted_permutation(name):
    """The MXFP8 dispatch takes its 32-row tiles in the order of their first
    row's token ("tile_order" in the workspace): a permutation of the tiles
    whose token buckets (1,024 over T) never decrease, all-padding tiles last.
    It is a processing order only; the outputs are checked by the parity tests."""
    cfg = small(name)
    c = Case(cfg, backward=False)
    run_forward(c, train=False)
    counts, offsets, poff, inv = c.route_views(1)
    T, k = cfg["T"], cfg["k"]
    ntiles = int(poff[-1]) // 32
    order = np.frombuffer(c.buffer(1, "tile_order").tobytes(), dtype=np.int32)[:ntiles]
    assert np.array_equal(np.sort(order), np.arange(ntiles))
    tok = np.full(ntiles, -1)                      # token of each tile's first row, -1: padding
    for e in range(cfg["E"]):
        for t in range(int(poff[e]) // 32, int(poff[e + 1]) // 32):
            local = t * 32 - int(poff[e])
            if local < counts[e]:
                tok[t] = inv[offsets[e] + local] // k
    key = np.where(tok < 0, 1023, tok * 1024 // T)
    assert np.all(np.diff(key[order]) >= 0)
