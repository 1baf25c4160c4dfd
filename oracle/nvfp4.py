"""NVFP4: 4-bit E2M1 elements with two-level scaling, written from the format's
public definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages name NVFP4 only to say the method has no NVFP4 path ("Mixture-of-
Kittens" wiki page, Key claims, MXFP8 bullet); the format and its
quantisation recipe are NVIDIA's published NVFP4 definition, which this module
restates:

* element: FP4 E2M1 -- 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit;
  magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no infinities, no NaN;
* every 16 consecutive elements along the reduction axis K share one scale
  stored as an FP8 E4M3 code (non-negative in use);
* a second-level fp32 scale per tensor, S_enc = (448 * 6) / amax(|tensor|)
  (1 for an all-zero tensor), maps the tensor's range so that the block
  scales use E4M3's range: the block scale is E4M3(amax_b / 6 * S_enc) and an
  element is stored as E2M1(x * S_enc / block_scale); it decodes to
  e2m1 * block_scale / S_enc.

Readings where the definition leaves a step open (each also listed in the
design notes):

* every scale computation is one IEEE fp32 operation at a time, in the
  order written above (amax_b / 6, then * S_enc; S_enc / block_scale, then
  x * that), with round-to-nearest-even -- so a device computing in fp32
  reaches the same codes bit for bit;
* E4M3 and E2M1 conversions round to nearest, ties to even, and saturate to
  the largest finite magnitude (448 and 6);
* a block whose scale code is 0 stores every element as a signed zero;
* two codes share a byte, element 2i in the low nibble, 2i + 1 in the high one.
"""
import numpy as np

from .numerics import e4m3_decode, e4m3_encode_bruteforce

NV_BLOCK = 16
E2M1_MAX = 6.0
E4M3_MAX = 448.0


# ----------------------------------------------------------------------------
# E2M1
# ----------------------------------------------------------------------------
def e2m1_decode_table():
    """float64 value of each of the 16 E2M1 codes (bit 3 = sign)."""
    vals = np.empty(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 0x8 else 1.0
        exp_field = (code >> 1) & 0x3
        man = code & 0x1
        if exp_field == 0:
            vals[code] = sign * man * 0.5                 # subnormal: (m/2) * 2**(1-1)
        else:
            vals[code] = sign * (1.0 + man / 2.0) * 2.0 ** (exp_field - 1)
    return vals


_E2M1 = e2m1_decode_table()
_E2M1_MAGS = _E2M1[:8]            # codes 0..7: the non-negative magnitudes, increasing


def e2m1_decode(codes):
    return _E2M1[np.asarray(codes, dtype=np.uint8) & 0xF]


def e2m1_encode(v):
    """Nearest E2M1 magnitude by exhaustive search over the 8 codes; among two
    equally near codes the one with an even mantissa bit wins; beyond 6 the
    nearest finite code (6) is taken; the sign bit is copied from the input."""
    v = np.asarray(v, dtype=np.float64)
    assert np.all(np.isfinite(v)), "E2M1 encoding expects finite inputs"
    a = np.minimum(np.abs(v), 2 * E2M1_MAX)[..., None]
    dist = np.abs(_E2M1_MAGS - a)
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best
    score = np.where(cand, np.where(np.arange(8) % 2 == 0, 0, 1), 2)
    mag = np.argmin(score, axis=-1).astype(np.uint8)
    return (mag | np.where(np.signbit(v), 0x8, 0).astype(np.uint8)).astype(np.uint8)


# ----------------------------------------------------------------------------
# two-level block quantisation
# ----------------------------------------------------------------------------
def f32(a):
    return np.asarray(a, dtype=np.float32)


def global_scale(amax):
    """S_enc = (448 * 6) / amax as one fp32 division; 1 for amax == 0."""
    amax = f32(amax)
    with np.errstate(divide="ignore"):
        s = f32(np.float32(E4M3_MAX * E2M1_MAX) / amax)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def nvfp4_quantize(v, s_enc, axis=-1):
    """Codes (uint8 0..15, one per element, v's shape) and E4M3 scale codes
    (blocked axis divided by 16) of ``v`` in blocks of 16 along ``axis``.

    ``v`` must hold fp32-representable values (bf16 tokens or weights, fp32
    activations); ``s_enc`` is the tensor's fp32 second-level scale.
    """
    v = np.asarray(v, dtype=np.float64)
    assert np.all(np.isfinite(v)), "NVFP4 quantisation expects finite inputs"
    assert np.array_equal(v.astype(np.float32).astype(np.float64), v), "inputs must be fp32 values"
    s_enc = np.float32(s_enc)
    v = np.moveaxis(v, axis, -1)
    K = v.shape[-1]
    assert K % NV_BLOCK == 0, "blocked axis must be a multiple of 16"
    b = f32(v.reshape(v.shape[:-1] + (K // NV_BLOCK, NV_BLOCK)))
    amax = np.abs(b).max(axis=-1)
    t = f32(f32(amax / np.float32(E2M1_MAX)) * s_enc)          # amax_b / 6, then * S_enc
    sf = e4m3_encode_bruteforce(t.astype(np.float64))
    sf_val = f32(e4m3_decode(sf))
    with np.errstate(divide="ignore"):
        inv = np.where(sf_val > 0, f32(s_enc / np.where(sf_val > 0, sf_val, np.float32(1))), np.float32(0))
    x = f32(b * inv[..., None])                                  # x * (S_enc / scale)
    codes = e2m1_encode(x.astype(np.float64)).reshape(v.shape)
    return np.moveaxis(codes, -1, axis), np.moveaxis(sf.astype(np.uint8), -1, axis)


def nvfp4_dequantize(codes, scales, s_enc, axis=-1):
    """float64 values e2m1 * scale / S_enc."""
    codes = np.moveaxis(np.asarray(codes, dtype=np.uint8), axis, -1)
    scales = np.moveaxis(np.asarray(scales, dtype=np.uint8), axis, -1)
    K = codes.shape[-1]
    vals = e2m1_decode(codes).reshape(codes.shape[:-1] + (K // NV_BLOCK, NV_BLOCK))
    out = (vals * e4m3_decode(scales)[..., None] / np.float64(np.float32(s_enc))).reshape(codes.shape)
    return np.moveaxis(out, -1, axis)


def nvfp4_roundtrip(v, s_enc, axis=-1):
    c, s = nvfp4_quantize(v, s_enc, axis=axis)
    return nvfp4_dequantize(c, s, s_enc, axis=axis)


def pack_pairs(codes):
    """Two codes per byte along the last axis: element 2i low nibble, 2i+1 high."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_pairs(packed):
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out
