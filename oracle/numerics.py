"""Number formats used by the layer, written from their definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 stored mantissa bits,
  i.e. 8 significant bits; round to nearest, ties to even.
* OCP FP8 E4M3 ("E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
  bits, no infinities, a single NaN magnitude (S.1111.111), largest finite
  magnitude 1.75 * 2**8 = 448, smallest normal 2**-6, subnormals m * 2**-9.
* OCP MX (Microscaling v1.0) MXFP8: blocks of 32 consecutive elements along
  the reduction axis share one E8M0 scale X = 2**e (byte e + 127); the
  shared exponent is floor(log2(amax)) minus the exponent of E4M3's largest
  normal (8); each element is E4M3(v / X), round-to-nearest-even,
  saturating.

The MXFP8 recipe (E4M3 codes, one E8M0 scale per 32 elements along K,
round-to-nearest-even, saturating) is what the configurations of the layer
state; the pages themselves only say MXFP8 is the default format and that
activation quantisation is fused into dispatch, the grouped GEMMs and SwiGLU
("Mixture-of-Kittens" wiki page, Key claims, MXFP8 bullet).

Readings where the definition leaves a case open:
* an all-zero block gets scale byte 0 (2**-127) and all-zero codes;
* inputs must be finite (NaN/Inf are rejected with an assertion);
* the sign of zero is kept (-0.0 encodes as 0x80).
"""
import numpy as np

MX_BLOCK = 32
E4M3_EMAX = 8          # exponent of the largest normal E4M3 value (448 = 1.75 * 2**8)
E4M3_MAX = 448.0
E8M0_BIAS = 127


# ----------------------------------------------------------------------------
# bfloat16
# ----------------------------------------------------------------------------
def bf16_round(a):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    Works binade by binade: a value in [2**(e-1), 2**e) is an integer
    multiple of 2**(e-8) when representable (8 significant bits); below the
    smallest normal 2**-126 the spacing stays 2**-133 (subnormals).  Values
    that round to 2**128 or beyond overflow to infinity.
    """
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)
    e_eff = np.maximum(e, -125)
    spacing_exp = e_eff - 8
    q = np.rint(np.ldexp(a, -spacing_exp))          # rint = round half to even
    r = np.ldexp(q, spacing_exp)
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, a), r)
    return r


def bf16_bits(a):
    """Bit pattern (uint16) of float64 values that are exact bfloat16 values."""
    a = np.asarray(a, dtype=np.float64)
    f32 = a.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), a, equal_nan=True), "not representable"
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits):
    """float64 values of bfloat16 bit patterns (uint16)."""
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# E4M3
# ----------------------------------------------------------------------------
def e4m3_decode_table():
    """float64 value of each of the 256 E4M3 codes (NaN for 0x7F and 0xFF)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        man = code & 0x7
        if exp_field == 15 and man == 7:
            vals[code] = np.nan
        elif exp_field == 0:
            vals[code] = sign * man * 2.0 ** -9          # subnormal: (m/8) * 2**(1-7)
        else:
            vals[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp_field - 7)
    return vals


_TABLE = e4m3_decode_table()
_MAGS = _TABLE[:127]            # codes 0..126: the finite non-negative magnitudes, increasing


def e4m3_decode(codes):
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def _apply_sign(mag_code, v):
    return (mag_code.astype(np.uint8) | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)).astype(np.uint8)


def e4m3_encode_bruteforce(v, chunk=1 << 15):
    """Nearest finite E4M3 magnitude by exhaustive search over all 127 codes.

    Among equally near codes the one with an even mantissa (even code) wins;
    magnitudes beyond 448 land on 448 (the nearest finite code), which is
    the saturating behaviour.  The sign bit is copied from the input.
    """
    v = np.asarray(v, dtype=np.float64)
    assert np.all(np.isfinite(v)), "E4M3 encoding expects finite inputs"
    # Beyond 2 * 448 every finite code is farther than 448 itself; clipping there
    # keeps the float64 distances exact without changing the nearest code.
    flat = np.minimum(np.abs(v.reshape(-1)), 2 * E4M3_MAX)
    out = np.empty(flat.shape, dtype=np.uint8)
    codes = np.arange(127)
    for s in range(0, flat.size, chunk):
        x = flat[s:s + chunk, None]
        dist = np.abs(_MAGS[None, :] - x)
        best = dist.min(axis=1, keepdims=True)
        cand = dist == best
        # prefer the even code among the (at most two) nearest candidates
        score = np.where(cand, np.where(codes[None, :] % 2 == 0, 0, 1), 2)
        out[s:s + chunk] = np.argmin(score, axis=1)
    return _apply_sign(out.reshape(v.shape), v)


def e4m3_encode(v):
    """Same result as :func:`e4m3_encode_bruteforce`, via the sorted code table.

    The two neighbouring magnitudes of |v| are located by binary search; the
    nearer one wins, ties go to the even code.
    """
    v = np.asarray(v, dtype=np.float64)
    assert np.all(np.isfinite(v)), "E4M3 encoding expects finite inputs"
    a = np.abs(v)
    hi = np.clip(np.searchsorted(_MAGS, a, side="left"), 1, 126)
    lo = hi - 1
    d_lo = a - _MAGS[lo]
    d_hi = _MAGS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo)
    mag = np.where(a >= E4M3_MAX, 126, mag)          # saturate
    return _apply_sign(mag, v)


# ----------------------------------------------------------------------------
# MXFP8 block quantisation
# ----------------------------------------------------------------------------
def mx_scale_exponent(amax):
    """Shared exponent of a block: floor(log2(amax)) - 8, clamped to [-127, 127].

    floor(log2(a)) is read exactly off frexp (a = f * 2**e, 0.5 <= f < 1
    gives floor(log2(a)) = e - 1).  amax == 0 gives -127.
    """
    amax = np.asarray(amax, dtype=np.float64)
    _, e = np.frexp(amax)
    es = (e - 1) - E4M3_EMAX
    es = np.where(amax > 0, es, -E8M0_BIAS)
    return np.clip(es, -E8M0_BIAS, E8M0_BIAS).astype(np.int64)


def mx_quantize(v, axis=-1):
    """MXFP8-quantise ``v`` in blocks of 32 consecutive elements along ``axis``.

    Returns (codes uint8 with v's shape, scale bytes uint8 with the blocked
    axis divided by 32).  The length along ``axis`` must be a multiple of 32.
    """
    v = np.asarray(v, dtype=np.float64)
    assert np.all(np.isfinite(v)), "MX quantisation expects finite inputs"
    v = np.moveaxis(v, axis, -1)
    K = v.shape[-1]
    assert K % MX_BLOCK == 0, "blocked axis must be a multiple of 32"
    b = v.reshape(v.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    es = mx_scale_exponent(np.abs(b).max(axis=-1))
    scaled = np.ldexp(b, -es[..., None])
    codes = e4m3_encode(scaled).reshape(v.shape)
    scales = (es + E8M0_BIAS).astype(np.uint8)
    return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis)


def mx_dequantize(codes, scales, axis=-1):
    """float64 values of MXFP8 codes with their per-32 E8M0 scale bytes."""
    codes = np.moveaxis(np.asarray(codes, dtype=np.uint8), axis, -1)
    scales = np.moveaxis(np.asarray(scales, dtype=np.uint8), axis, -1)
    K = codes.shape[-1]
    vals = e4m3_decode(codes).reshape(codes.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    out = np.ldexp(vals, scales.astype(np.int64)[..., None] - E8M0_BIAS).reshape(codes.shape)
    return np.moveaxis(out, -1, axis)


def mx_roundtrip(v, axis=-1):
    """Dequantised value of the MXFP8 quantisation of ``v`` (float64)."""
    c, s = mx_quantize(v, axis=axis)
    return mx_dequantize(c, s, axis=axis)
