"""Pins for oracle/numerics.py against definitions, library casts and brute force."""
import os

import numpy as np
import pytest
import torch

from oracle import numerics as nx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = nx.bf16_from_bits(bits)
    return v[np.isfinite(v)]


def test_e4m3_table_matches_golden_definition():
    table = nx.e4m3_decode_table()
    n = 0
    with open(os.path.join(GOLDEN, "e4m3_special_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            code, val = line.split()
            code = int(code, 16)
            want = float(val)
            if np.isnan(want):
                assert np.isnan(table[code])
            else:
                assert table[code] == want and np.signbit(table[code]) == np.signbit(want), hex(code)
            n += 1
    assert n >= 15


def test_e4m3_table_matches_torch_float8_cast():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    table = nx.e4m3_decode_table()
    assert np.array_equal(np.isnan(ref), np.isnan(table))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], table[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(table[ok]))


@pytest.mark.parametrize("shift", [-12, -6, 0, 3, 8])
def test_e4m3_encode_matches_bruteforce_exhaustive(shift):
    v = np.ldexp(all_finite_bf16(), shift)
    v = v[np.isfinite(v)]
    a = nx.e4m3_encode(v)
    b = nx.e4m3_encode_bruteforce(v)
    assert np.array_equal(a, b)


def test_e4m3_encode_matches_torch_cast_in_range():
    # torch's float -> float8_e4m3fn cast is round-to-nearest-even but maps
    # overflow to NaN, so compare on |v| <= 448 only (saturation is pinned below).
    v = all_finite_bf16()
    for shift in (-10, -4, 0, 4):
        s = np.ldexp(v, shift)
        s = s[np.isfinite(s) & (np.abs(s) <= 448.0)]
        ref = torch.from_numpy(s.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(nx.e4m3_encode(s), ref)


def test_e4m3_saturates_and_keeps_sign():
    v = np.array([448.0, 449.0, 464.0, 480.0, 1e6, -1e6, -0.0, 0.0, -1e-9])
    c = nx.e4m3_encode(v)
    assert list(c) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00, 0x80]


def test_e4m3_ties_go_to_even():
    # 1.0625 is halfway between 1.0 (0x38) and 1.125 (0x39): even code wins.
    # 1.1875 is halfway between 1.125 (0x39) and 1.25 (0x3A): even code wins.
    assert list(nx.e4m3_encode(np.array([1.0625, 1.1875, -1.0625]))) == [0x38, 0x3A, 0xB8]
    # halfway between the two smallest subnormals
    assert nx.e4m3_encode(np.array([1.5 * 2.0 ** -9]))[0] == 0x02
    assert nx.e4m3_encode(np.array([0.5 * 2.0 ** -9]))[0] == 0x00


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    a = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(20000) * 1e37).astype(np.float32),
    ])
    # exact midpoints between neighbouring bf16 values (ties)
    bits = rng.integers(0, 1 << 16, 20000).astype(np.uint32)
    mids = ((bits << 16) | 0x8000).view(np.float32)
    a = np.concatenate([a, mids[np.isfinite(mids)]])
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = nx.bf16_round(a.astype(np.float64))
    assert np.array_equal(ref, got)


def test_bf16_bits_roundtrip():
    v = all_finite_bf16()
    assert np.array_equal(nx.bf16_from_bits(nx.bf16_bits(v)), v)


def test_mx_closed_forms():
    blk = np.zeros(32)
    blk[0] = 1.0
    c, s = nx.mx_quantize(blk)
    assert s[0] == 119 and c[0] == 0x78 and np.all(c[1:] == 0)         # 1 = 256 * 2**-8
    blk[0] = 448.0
    c, s = nx.mx_quantize(blk)
    assert s[0] == 127 and c[0] == 0x7E                                  # scale 2**0
    blk[0] = 511.0                                                       # floor(log2) = 8 -> scale 1, saturates
    c, s = nx.mx_quantize(blk)
    assert s[0] == 127 and c[0] == 0x7E
    blk[0] = -3.0 * 2.0 ** -130                                          # scale clamps at 2**-127
    c, s = nx.mx_quantize(blk)
    assert s[0] == 0 and c[0] == (0x80 | nx.e4m3_encode(np.array([3.0 * 2.0 ** -3]))[0])
    c, s = nx.mx_quantize(np.zeros(64))
    assert np.all(s == 0) and np.all(c == 0)


def test_mx_error_bound_random():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-20, 20, (64, 1)))
    c, s = nx.mx_quantize(v, axis=1)
    deq = nx.mx_dequantize(c, s, axis=1)
    es = (s.astype(np.int64) - 127).repeat(32, axis=1)
    scaled = np.abs(v) / 2.0 ** es
    # element bound: half a unit in the 3-bit mantissa (relative 2**-4) for normal
    # codes, 2**-10 absolute below the smallest normal, saturation above 448.
    bound = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** (es - 10))
    sat = scaled > 448.0
    bound = np.where(sat, np.abs(v) - 448.0 * 2.0 ** es, bound)
    assert np.all(np.abs(deq - v) <= bound * (1 + 1e-12))
    # the block maximum always lands in [256, 448] after scaling
    amax = np.abs(v).reshape(64, 8, 32).max(-1)
    sc = amax / 2.0 ** (s.astype(np.int64) - 127)
    assert np.all((sc >= 256) & (sc < 512))


def test_mx_axis_consistency():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 96))
    c0, s0 = nx.mx_quantize(v, axis=0)
    c1, s1 = nx.mx_quantize(v.T, axis=1)
    assert np.array_equal(c0, c1.T) and np.array_equal(s0, s1.T)
