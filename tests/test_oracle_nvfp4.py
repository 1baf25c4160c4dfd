"""Pins for oracle/nvfp4.py (the NVFP4 variant of the expert GEMMs): the E2M1
table against the format's defining values, the encoder's ties and
saturation, exact round trips of representable blocks, the second-level
scale's closed forms, and exact expert products on representable operands."""
import os

import numpy as np
import pytest

from oracle import moe as om
from oracle import numerics as nx
from oracle import nvfp4 as nv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_values.txt")


def test_e2m1_table_matches_the_format_definition():
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        code, val = line.split()
        v = nv.e2m1_decode(int(code, 16))
        assert v == float(val) and np.signbit(v) == val.startswith("-")


@pytest.mark.parametrize("x,code", [
    (0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5.0, 0x6),   # ties -> even
    (0.26, 0x1), (1.3, 0x3), (2.6, 0x5), (5.1, 0x7),                                       # just past a tie
    (6.0, 0x7), (7.0, 0x7), (1e6, 0x7),                                                     # saturation
    (-0.0, 0x8), (-1.6, 0xb), (-9.0, 0xf), (0.0, 0x0),
])
def test_e2m1_encode_ties_saturation_sign(x, code):
    assert int(nv.e2m1_encode(x)) == code


def test_e2m1_encode_is_nearest_on_a_fine_grid():
    v = np.linspace(-7.0, 7.0, 14001)
    got = nv.e2m1_decode(nv.e2m1_encode(v))
    err = np.abs(got - np.clip(v, -6, 6))
    mags = np.abs(nv._E2M1_MAGS)
    best = np.abs(mags[None, :] - np.minimum(np.abs(v), 6)[:, None]).min(axis=1)
    assert np.allclose(err, best)


def test_global_scale_closed_forms():
    assert nv.global_scale(6.0) == np.float32(448.0)
    assert nv.global_scale(2688.0) == np.float32(1.0)
    assert nv.global_scale(0.0) == np.float32(1.0)
    assert nv.global_scale(3.0) == np.float32(896.0)


def test_representable_blocks_round_trip_exactly():
    """Blocks built as e2m1 * scale with one element at +-6 * scale: the block
    scale is recovered exactly (amax / 6 = scale) and so are the codes."""
    rng = np.random.default_rng(0)
    nb = 64
    codes = rng.integers(0, 16, (nb, 16)).astype(np.uint8)
    codes[:, 3] = np.where(rng.random(nb) < 0.5, 0x7, 0xF)        # each block holds +-6
    sf = rng.integers(0x08, 0x7F, nb).astype(np.uint8)           # normal E4M3 scales
    vals = nv.e2m1_decode(codes) * nx.e4m3_decode(sf)[:, None]
    c, s = nv.nvfp4_quantize(vals.reshape(1, -1), 1.0, axis=1)
    assert np.array_equal(s.reshape(-1), sf)
    same = (c.reshape(nb, 16) == codes) | ((codes & 7) == 0) & ((c.reshape(nb, 16) & 7) == 0)
    assert same.all()
    assert np.array_equal(nv.nvfp4_roundtrip(vals.reshape(1, -1), 1.0, axis=1).reshape(nb, 16), vals)


def test_second_level_scale_puts_the_largest_block_at_448():
    rng = np.random.default_rng(1)
    v = nx.bf16_round(rng.standard_normal((8, 64)) * 1e-3)
    v[5, 17] = 0.375                                            # the tensor's amax, alone in its block
    s = nv.global_scale(np.abs(v).max())
    c, sf = nv.nvfp4_quantize(v, s, axis=1)
    assert sf[5, 1] == 0x7E and nx.e4m3_decode(0x7E) == 448.0
    assert nv.e2m1_decode(c[5, 17]) == 6.0
    # all scales stay finite codes, and the round trip is within half an E2M1 step per block
    rt = nv.nvfp4_roundtrip(v, s, axis=1)
    step = nx.e4m3_decode(sf).repeat(16, axis=1) / np.float64(s)
    assert np.all(np.abs(rt - v) <= 1.0 * step + 1e-30)


def test_zero_blocks_and_signs():
    v = np.zeros((2, 32))
    v[1, :16] = -0.0
    v[1, 16:] = [-1.0] + [0.0] * 15
    c, s = nv.nvfp4_quantize(v, 1.0, axis=1)
    assert np.all(s[0] == 0) and np.all(c[0] == 0)
    assert s[1, 0] == 0 and np.all(c[1, :16] == 0x8)               # -0 keeps its sign
    # amax 1 with S_enc = 1: the block scale is E4M3(1/6) = 0.171875, -1 becomes -6 * 0.171875
    assert s[1, 1] == 0x23 and c[1, 16] == 0xF and nv.e2m1_decode(c[1, 16]) * nx.e4m3_decode(s[1, 1]) == -1.03125


def test_pack_pairs_low_nibble_first():
    codes = np.array([[0x1, 0xF, 0x7, 0x8]], dtype=np.uint8)
    p = nv.pack_pairs(codes)
    assert p.tolist() == [[0xF1, 0x87]]
    assert np.array_equal(nv.unpack_pairs(p), codes)


def test_nvfp4_expert_forward_exact_when_operands_representable():
    """X representable in NVFP4 along d under the whole-x second-level scale,
    weights representable along their K under their own: G and U equal the
    unquantised products, while quantising along the other axis would not."""
    rng = np.random.default_rng(2)
    n, d, m = 16, 64, 32

    def rep(rows, cols, S, rng):
        """e2m1 * scale / S per 16-block, each block holding +-6 and one block's
        scale 448, so the tensor's second-level scale is S (a power of two) and
        every block scale is recovered exactly."""
        codes = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
        codes[:, ::16] = 0x7
        sf = rng.integers(0x20, 0x70, (rows, cols // 16)).astype(np.uint8)
        sf[0, 0] = 0x7E
        return nv.e2m1_decode(codes) * nx.e4m3_decode(sf).repeat(16, axis=1) / S

    X, W_gu, W_dn = rep(n, d, 2.0 ** 8, rng), rep(2 * m, d, 2.0 ** 13, rng), rep(d, m, 2.0 ** 12, rng)
    for A, S in ((X, 2.0 ** 8), (W_gu, 2.0 ** 13), (W_dn, 2.0 ** 12)):
        s = nv.global_scale(np.abs(A).max())
        assert s == np.float32(S)
        assert np.array_equal(nv.nvfp4_roundtrip(A, s, axis=1), A)
        assert not np.array_equal(nv.nvfp4_roundtrip(A, s, axis=0), A)
    res = om.expert_forward(X, W_gu, W_dn, "nvfp4")
    assert np.array_equal(res["G"], X @ W_gu[:m].T) and np.array_equal(res["U"], X @ W_gu[m:].T)


def test_nvfp4_forward_close_to_exact_and_needs_the_whole_x_scale():
    rng = np.random.default_rng(3)
    T, d, m, E, k = 40, 64, 32, 4, 2
    x = nx.bf16_round(rng.standard_normal((T, d)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    experts = [(nx.bf16_round(rng.standard_normal((2 * m, d)) / 8), nx.bf16_round(rng.standard_normal((d, m)) / 6))
               for _ in range(E)]
    y64, _ = om.forward(x, logits, experts, k, "fp64")
    y, _ = om.forward(x, logits, experts, k, "nvfp4")
    assert np.linalg.norm(y - y64) / np.linalg.norm(y64) < 0.3
    # a token subset with the whole x's scale gives the same rows as the full forward
    sub = np.array([3, 7, 21])
    y_sub, _ = om.forward(x[sub], logits[sub], experts, k, "nvfp4",
                          x_scale=nv.global_scale(np.abs(x).max()))
    assert np.array_equal(y_sub, y[sub])
    with pytest.raises(NotImplementedError):
        om.prepare_expert(experts[0][0], experts[0][1], "nvfp4", backward=True)


def test_nvfp4_h_quantised_along_m_with_unit_second_level_scale():
    """h = 64 * U exactly (a gate of 64 makes silu(G) = G), with U = x[:, 16:16+m]
    built so that h is NVFP4-representable along m under second-level scale 1
    and not along rows: o then equals the unquantised product bit for bit."""
    rng = np.random.default_rng(4)
    n, d, m = 32, 64, 32
    S = 2.0 ** 8                                     # x's second-level scale (power of two)
    x = np.zeros((n, d))
    x[:, 0] = 1.0                                    # = 4 * (64 / 256): code 4.0, block scale 64
    x[:, 1] = 1.5                                    # the block's amax: 6 * 64 / 256
    codes = rng.integers(0, 16, (n, m)).astype(np.uint8)
    codes[:, ::16] = 0x7
    sfv = (0x30 + 8 * rng.integers(0, 4, (n, m // 16))).astype(np.uint8)   # scales 2**-1 .. 2**2, per row
    V = nv.e2m1_decode(codes) * nx.e4m3_decode(sfv).repeat(16, axis=1) / S
    x[:, 16:16 + m] = V
    x[0, 48:64] = 0.0
    x[0, 48] = 6.0 * 448.0 / S                       # one block at scale 448: x's amax, S_enc = S
    W_gu = np.zeros((2 * m, d))
    W_gu[:m, 0] = 64.0                               # gate: G = 64 * x[:, 0] = 64
    W_gu[m + np.arange(m), 16 + np.arange(m)] = 1.0  # up: U = x[:, 16:16+m]
    W_dn = nv.e2m1_decode(rng.integers(0, 16, (d, m)).astype(np.uint8))
    W_dn[:, ::16] = 6.0
    h = 64.0 * V
    assert nv.global_scale(np.abs(x).max()) == np.float32(S)
    assert np.array_equal(nv.nvfp4_roundtrip(x, S, axis=1), x)
    assert np.array_equal(nv.nvfp4_roundtrip(h, 1.0, axis=1), h)
    assert not np.array_equal(nv.nvfp4_roundtrip(h, 1.0, axis=0), h)
    res = om.expert_forward(x, W_gu, W_dn, "nvfp4")
    assert np.array_equal(res["G"], np.full((n, m), 64.0)) and np.array_equal(res["U"], V)
    assert np.array_equal(res["o"], nx.bf16_round(h @ W_dn.T))
