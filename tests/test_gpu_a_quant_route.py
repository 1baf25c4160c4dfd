"""GPU parity of the integer / byte parts of the path: MXFP8 quantisation
(codes and scales bit-exact), router top-k and the schedule (bit-exact), the
softmax weights (fp32 vs fp64 within a derived bound)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import unpack_tiled_scales
from oracle import moe as om
from oracle import numerics as nx

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    import mixture_experts_layer_device_gb300 as m
    return m


def _quant(pkg, w, transpose):
    B, rows, cols = w.shape
    n = B * rows * cols
    codes = torch.empty(n, dtype=torch.uint8, device="cuda")
    sf = torch.empty(n // 32, dtype=torch.uint8, device="cuda")
    pkg.check(pkg.moe_quantize_mx(w, B, rows, cols, transpose, codes, sf))
    torch.cuda.synchronize()
    return codes.cpu().numpy(), sf.cpu().numpy()


def edge_values(rng, shape):
    v = rng.standard_normal(shape).astype(np.float32)
    v[0, 0, :64] = 0.0                                   # all-zero blocks
    v[0, 1, :32] = rng.standard_normal(32) * 1e-39       # subnormal-only block
    v[0, 2, :32] = rng.uniform(-1.0, 1.0, 32) * 3e38     # near the top of the range
    v[0, 3, :32] = np.float32(448.0) * 2.0 ** rng.integers(-20, 20)
    v[0, 3, 5] = -v[0, 3, 5]
    v[0, 4, :] = -0.0
    v[0, 5, :32] = np.ldexp(1.0, rng.integers(-140, 120, 32))   # wide per-element exponent spread
    return v


@pytest.mark.parametrize("transpose", [0, 1])
def test_quantize_mx_bit_exact(pkg, transpose):
    rng = np.random.default_rng(0)
    v = edge_values(rng, (2, 256, 384))
    w = torch.from_numpy(v).to(torch.bfloat16)
    codes, sf = _quant(pkg, w.cuda(), transpose)
    ref = mi.to_f64(w)
    c_ref, s_ref = om.quantize_weights(ref, transpose=bool(transpose))
    B, rows, cols = c_ref.shape
    assert np.array_equal(codes.reshape(B * rows, cols), c_ref.reshape(B * rows, cols))
    assert np.array_equal(sf.reshape(B * rows, cols // 32), s_ref.reshape(B * rows, cols // 32))   # canonical


@pytest.mark.parametrize("shape", [(2, 256, 384), (3, 384, 128)])
def test_quantize_mx_both_orientations_bit_exact(pkg, shape):
    """One read of the masters gives both operand orientations, each
    bit-identical to the oracle's quantisation of that orientation."""
    rng = np.random.default_rng(1)
    v = edge_values(rng, shape)
    w = torch.from_numpy(v).to(torch.bfloat16)
    B, rows, cols = shape
    n = B * rows * cols
    out = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(2)]
    osf = [torch.empty(n // 32, dtype=torch.uint8, device="cuda") for _ in range(2)]
    pkg.check(pkg.moe_quantize_mx_both(w.cuda(), B, rows, cols, out[0], osf[0], out[1], osf[1]))
    torch.cuda.synchronize()
    ref = mi.to_f64(w)
    for transpose in (0, 1):
        c_ref, s_ref = om.quantize_weights(ref, transpose=bool(transpose))
        Bq, r, c = c_ref.shape
        assert np.array_equal(out[transpose].cpu().numpy().reshape(Bq * r, c), c_ref.reshape(Bq * r, c))
        assert np.array_equal(osf[transpose].cpu().numpy().reshape(Bq * r, c // 32),
                              s_ref.reshape(Bq * r, c // 32))


def test_quantize_mx_exhaustive_bf16_patterns(pkg):
    # every finite bf16 bit pattern, in blocks that also carry a large element
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = nx.bf16_from_bits(bits)
    vals = vals[np.isfinite(vals)]
    n = (vals.size + 127) // 128 * 128 * 128
    arr = np.zeros(n)
    arr[:vals.size] = vals
    w = torch.from_numpy(arr.reshape(1, -1, 128).astype(np.float32)).to(torch.bfloat16)
    codes, sf = _quant(pkg, w.cuda(), 0)
    c_ref, s_ref = nx.mx_quantize(mi.to_f64(w)[0], axis=1)
    assert np.array_equal(codes.reshape(c_ref.shape), c_ref)
    assert np.array_equal(sf.reshape(s_ref.shape), s_ref)


@pytest.mark.parametrize("rows,K", [(128, 128), (384, 512), (1024, 7168)])
def test_prepare_and_canonical_scales_bit_exact(pkg, rows, K):
    """moe_prepare_scales is the permutation the prepared layout defines (index
    arithmetic written out in the tests' helper) and moe_canonical_scales its
    inverse; a same-pointer call and shapes off the 128 grid are refused."""
    rng = np.random.default_rng(rows + K)
    canon = rng.integers(0, 256, (rows, K // 32), dtype=np.uint8)
    src = torch.from_numpy(canon).cuda()
    prep = torch.empty(rows * K // 32, dtype=torch.uint8, device="cuda")
    back = torch.empty_like(src)
    pkg.check(pkg.moe_prepare_scales(src, rows, K, prep))
    pkg.check(pkg.moe_canonical_scales(prep, rows, K, back))
    torch.cuda.synchronize()
    p = prep.cpu().numpy()
    assert np.array_equal(unpack_tiled_scales(p, rows, K), canon)
    assert np.array_equal(back.cpu().numpy(), canon)
    assert sorted(p.tolist()) == sorted(canon.reshape(-1).tolist())
    assert pkg.moe_prepare_scales(src, rows, K, src) == -1
    assert pkg.moe_prepare_scales(src, rows + 32, K, prep) == -2
    assert pkg.moe_canonical_scales(prep, rows, K + 32, back) == -2


@pytest.mark.parametrize("backward", [False, True])
def test_prepare_weights_equals_quantise_then_prepare(pkg, backward):
    """moe_prepare_weights (the layer's S0, one read per master, prepared scales
    written directly) gives the bytes of moe_quantize_weights followed by
    moe_prepare_scales, in both orientations."""
    E, d, m = 3, 512, 256
    c = pkg.config(64, d, m, E, 2, 0, "mxfp8", pkg.MOE_FLAG_BACKWARD if backward else 0)
    rng = np.random.default_rng(9)
    gu = torch.from_numpy(edge_values(rng, (E, 2 * m, d))).to(torch.bfloat16).cuda()
    dn = torch.from_numpy(edge_values(rng, (E, d, m))).to(torch.bfloat16).cuda()
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device="cuda")
    n_gu, n_dn = E * 2 * m * d, E * d * m
    out = dict(gu=u8(n_gu), gu_scale=u8(n_gu // 32), dn=u8(n_dn), dn_scale=u8(n_dn // 32))
    if backward:
        out.update(gu_t=u8(n_gu), gu_t_scale=u8(n_gu // 32), dn_t=u8(n_dn), dn_t_scale=u8(n_dn // 32))
    pkg.check(pkg.moe_prepare_weights(c, gu, dn, **out))
    for key, w, rows, cols in (("gu", gu, 2 * m, d), ("dn", dn, d, m)):
        for t in ((0, 1) if backward else (0,)):
            name = key + ("_t" if t else "")
            codes, sc, prep = u8(E * rows * cols), u8(E * rows * cols // 32), u8(E * rows * cols // 32)
            pkg.check(pkg.moe_quantize_weights(c, w, rows, cols, t, codes, sc))
            pkg.check(pkg.moe_prepare_scales(sc, E * (cols if t else rows), rows if t else cols, prep))
            assert torch.equal(out[name], codes), name
            assert torch.equal(out[name + "_scale"], prep), name + "_scale"
    # one backward operand alone is refused
    assert pkg.moe_prepare_weights(c, gu, dn, out["gu"], out["gu_scale"], out["dn"], out["dn_scale"],
                                   out["gu"], out["gu_scale"], None, None) == -1


def _route(pkg, logits, k):
    T, E = logits.shape
    cfg = pkg.config(T, 256, 128, E, k)
    ws = torch.empty(pkg.moe_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    pkg.check(pkg.moe_route(cfg, logits.cuda(), idx, w, counts, offsets, perm, ws))
    assert pkg.moe_get_status(ws) == 0
    return [t.cpu().numpy() for t in (idx, w, counts, offsets, perm)]


def _check_route(pkg, logits, k):
    idx, w, counts, offsets, perm = _route(pkg, logits, k)
    l = logits.numpy()
    ridx, rw = om.route(l, k)
    rc, ro, rp, _ = om.schedule(ridx, l.shape[1])
    assert np.array_equal(idx, ridx)
    assert np.array_equal(counts, rc) and np.array_equal(offsets, ro) and np.array_equal(perm, rp)
    # fp32 softmax over k values vs fp64: expf error (a few ulp), k-term sum and a
    # division -> |err| <= (4 + k) * 2**-24 relative to the largest weight (<= 1).
    assert np.abs(w - rw).max() <= (4 + k) * 2.0 ** -24 * 2
    assert np.allclose(w.sum(1), 1.0, atol=(k + 2) * 2.0 ** -23)


@pytest.mark.parametrize("name", mi.ORDER)
def test_route_full_size_bit_exact(pkg, name):
    cfg = mi.WORKLOADS[name]
    _check_route(pkg, mi.logits(cfg), cfg["k"])


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (37, 5, 5), (300, 33, 7), (1000, 512, 16), (129, 1024, 3)])
def test_route_ragged_shapes(pkg, T, E, k):
    g = torch.Generator().manual_seed(T * 7 + E)
    _check_route(pkg, torch.randn((T, E), generator=g), k)


def test_route_ties_and_degenerate_loads(pkg):
    T, E, k = 700, 40, 6
    g = torch.Generator().manual_seed(5)
    l = torch.round(torch.randn((T, E), generator=g) * 2) / 2     # many exact ties
    l[10] = 0.0                                                   # an all-equal row
    l[:, 7] += 100.0                                              # an expert with every token
    l[:, 30:] -= 100.0                                            # experts that no token picks
    l[20, :] = -0.0
    l[21, ::2] = 0.0
    _check_route(pkg, l.contiguous(), k)


@pytest.mark.parametrize("blocks_along_rows", [0, 1])
def test_quantize_weights_layer_entry_bit_exact(pkg, blocks_along_rows):
    """moe_quantize_weights: the layer's stacked expert masters (cfg.E of
    them) in either operand orientation, bit-identical to the oracle; a BF16
    config is refused."""
    E, rows, cols = 3, 256, 512
    c = pkg.config(64, cols, rows // 2, E, 2, 0, "mxfp8", 0)
    rng = np.random.default_rng(5)
    w = torch.from_numpy(edge_values(rng, (E, rows, cols))).to(torch.bfloat16)
    wg = w.cuda()
    codes = torch.empty(E * rows * cols, dtype=torch.uint8, device="cuda")
    sf = torch.empty(E * rows * cols // 32, dtype=torch.uint8, device="cuda")
    pkg.check(pkg.moe_quantize_weights(c, wg, rows, cols, blocks_along_rows, codes, sf))
    torch.cuda.synchronize()
    c_ref, s_ref = om.quantize_weights(mi.to_f64(w), transpose=bool(blocks_along_rows))
    B, r2, c2 = c_ref.shape
    assert np.array_equal(codes.cpu().numpy().reshape(B * r2, c2), c_ref.reshape(B * r2, c2))
    assert np.array_equal(sf.cpu().numpy().reshape(B * r2, c2 // 32), s_ref.reshape(B * r2, c2 // 32))
    cb = pkg.config(64, cols, rows // 2, E, 2, 0, "bf16", 0)
    assert pkg.moe_quantize_weights(cb, wg, rows, cols, blocks_along_rows, codes, sf) == -1  # MOE_ERR_ARG
