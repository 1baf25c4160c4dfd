"""Pins for oracle/moe.py: brute force, invariants, closed forms, reductions to
plain formulas, and central finite differences of the backward pass."""
import numpy as np
import pytest

from oracle import moe as om
from oracle import numerics as nx


def rand_layer(rng, T, d, m, E, k, ms=0, bf16=True):
    f = nx.bf16_round if bf16 else (lambda a: a)
    x = f(rng.standard_normal((T, d)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    W_gu = f(rng.standard_normal((E, 2 * m, d)) / np.sqrt(d))
    W_dn = f(rng.standard_normal((E, d, m)) / np.sqrt(m))
    experts = [(W_gu[e], W_dn[e]) for e in range(E)]
    shared = None
    if ms:
        shared = (f(rng.standard_normal((2 * ms, d)) / np.sqrt(d)), f(rng.standard_normal((d, ms)) / np.sqrt(ms)))
    return x, logits, experts, shared


# ---------------------------------------------------------------- route
def brute_route(logits, k):
    T, E = logits.shape
    idx = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        taken = []
        for _ in range(k):
            best = None
            for e in range(E):
                if e in taken:
                    continue
                if best is None or float(logits[t, e]) > float(logits[t, best]):
                    best = e
            taken.append(best)
        idx[t] = taken
    return idx


@pytest.mark.parametrize("ties", [False, True])
def test_route_matches_bruteforce(ties):
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((64, 12)).astype(np.float32)
    if ties:
        logits = (np.round(logits * 2) / 2).astype(np.float32)
        logits[5] = 0.25
        logits[6, :] = logits[6, 0]
    idx, w = om.route(logits, 4)
    assert np.array_equal(idx, brute_route(logits, 4))
    if ties:
        assert list(idx[5]) == [0, 1, 2, 3]


def test_route_weights_equal_full_softmax_renormalised():
    rng = np.random.default_rng(4)
    logits = (rng.standard_normal((50, 16)) * 3).astype(np.float32)
    idx, w = om.route(logits, 5)
    l = logits.astype(np.float64)
    p = np.exp(l - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    sel = np.take_along_axis(p, idx, 1)
    assert np.allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-13, atol=0)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)                 # slot order = descending weight


# ---------------------------------------------------------------- schedule
def brute_schedule(idx, E):
    flat = list(np.asarray(idx).reshape(-1))
    row = 0
    perm = [None] * len(flat)
    for e in range(E):
        for i, ei in enumerate(flat):
            if ei == e:
                perm[i] = row
                row += 1
    return np.array(perm)


def test_schedule_invariants_and_bruteforce():
    rng = np.random.default_rng(5)
    T, E, k = 97, 9, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 4] += 5.0           # one hot expert
    logits[:, 7] -= 9.0           # one (almost surely) empty expert
    idx, _ = om.route(logits, k)
    counts, offsets, perm, inv = om.schedule(idx, E)
    R = T * k
    assert counts.sum() == R and offsets[-1] == R and offsets[0] == 0
    assert counts[7] == 0 and counts[4] == T
    assert np.array_equal(np.sort(perm), np.arange(R))
    assert np.array_equal(perm[inv], np.arange(R)) and np.array_equal(inv[perm], np.arange(R))
    flat = idx.reshape(-1)
    for e in range(E):
        rows = inv[offsets[e]:offsets[e + 1]]
        assert np.all(flat[rows] == e) and np.all(np.diff(rows) > 0)
    assert np.array_equal(perm, brute_schedule(idx, E))


# ---------------------------------------------------------------- forward
def ffn(X, W_gu, W_dn):
    m = W_gu.shape[0] // 2
    G = X @ W_gu[:m].T
    U = X @ W_gu[m:].T
    return ((G / (1 + np.exp(-G))) * U) @ W_dn.T


def test_sparse_equals_dense_masked_sum():
    rng = np.random.default_rng(6)
    T, d, m, E, k, ms = 23, 16, 8, 6, 2, 4
    x, logits, experts, shared = rand_layer(rng, T, d, m, E, k, ms, bf16=False)
    y, _ = om.forward(x, logits, experts, k, "fp64", shared=shared)
    # dense: every expert on every token, masked by the top-k choice
    l = logits.astype(np.float64)
    dense = np.zeros((T, d))
    for e in range(E):
        out = ffn(x, *experts[e])
        for t in range(T):
            order = sorted(range(E), key=lambda i: (-l[t, i], i))[:k]
            if e in order:
                z = np.exp(l[t, order] - l[t, order[0]])
                dense[t] += (z[order.index(e)] / z.sum()) * out[t]
    dense += ffn(x, *shared)
    assert np.abs(y - dense).max() <= 1e-12 * np.abs(dense).max()


def test_k_equals_E_uniform_logits_is_expert_average():
    rng = np.random.default_rng(7)
    T, d, m, E = 11, 8, 4, 5
    x, _, experts, _ = rand_layer(rng, T, d, m, E, E, bf16=False)
    logits = np.zeros((T, E), dtype=np.float32)
    y, saved = om.forward(x, logits, experts, E, "fp64")
    avg = sum(ffn(x, *experts[e]) for e in range(E)) / E
    assert np.allclose(y, avg, rtol=1e-12, atol=1e-13)
    assert np.array_equal(saved["idx"], np.tile(np.arange(E), (T, 1)))


@pytest.mark.parametrize("fmt", ["fp64", "bf16"])
def test_single_expert_is_plain_swiglu_ffn(fmt):
    rng = np.random.default_rng(8)
    x, logits, experts, _ = rand_layer(rng, 13, 16, 8, 1, 1)
    y, _ = om.forward(x, logits, experts, 1, fmt)
    ref = ffn(x, *experts[0])
    if fmt == "fp64":
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-13)
    else:
        W_gu, W_dn = experts[0]
        G, U = x @ W_gu[:8].T, x @ W_gu[8:].T
        h = nx.bf16_round(G / (1 + np.exp(-G)) * U)
        assert np.array_equal(y, nx.bf16_round(nx.bf16_round(h @ W_dn.T)))


def test_mx_forward_exact_when_operands_representable():
    """With x and weights exactly representable in MXFP8 along their K axes, the
    gate/up products equal the unquantised ones exactly; quantising along a wrong
    axis would not (the per-row magnitudes differ wildly)."""
    rng = np.random.default_rng(9)
    n, d, m = 5, 64, 32
    mant = lambda shape: (rng.integers(8, 15, shape) * rng.choice([-1, 1], shape)) / 8.0
    X = mant((n, d)) * 2.0 ** rng.integers(-3, 4, (n, 1))
    W_gu = mant((2 * m, d)) * 2.0 ** rng.integers(-9, 9, (2 * m, 1))
    W_dn = mant((d, m)) * 2.0 ** rng.integers(-9, 9, (d, 1))
    assert np.array_equal(nx.mx_roundtrip(X, 1), X) and np.array_equal(nx.mx_roundtrip(W_gu, 1), W_gu)
    assert not np.array_equal(nx.mx_roundtrip(W_gu, 0), W_gu)
    res = om.expert_forward(X, W_gu, W_dn, "mxfp8")
    assert np.array_equal(res["G"], X @ W_gu[:m].T) and np.array_equal(res["U"], X @ W_gu[m:].T)


@pytest.mark.parametrize("fmt,tol", [("bf16", 2e-2), ("mxfp8", 8e-2)])
def test_rounded_formats_close_to_exact(fmt, tol):
    rng = np.random.default_rng(10)
    T, d, m, E, k = 40, 64, 32, 4, 2
    x, logits, experts, _ = rand_layer(rng, T, d, m, E, k)
    y64, _ = om.forward(x, logits, experts, k, "fp64")
    y, _ = om.forward(x, logits, experts, k, fmt)
    assert np.linalg.norm(y - y64) / np.linalg.norm(y64) < tol


def test_quantize_weights_transpose():
    rng = np.random.default_rng(11)
    W = nx.bf16_round(rng.standard_normal((3, 64, 96)))
    c, s = om.quantize_weights(W, transpose=True)
    assert c.shape == (3, 96, 64) and s.shape == (3, 96, 2)
    c2, s2 = nx.mx_quantize(W[1].T, axis=1)
    assert np.array_equal(c[1], c2) and np.array_equal(s[1], s2)


# ---------------------------------------------------------------- backward
def _loss(x, logits, experts, k, shared, dy):
    y, _ = om.forward(x, logits, experts, k, "fp64", shared=shared)
    return float((y * dy).sum())


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(12)
    T, d, m, E, k, ms = 7, 8, 4, 4, 2, 4
    x, logits, experts, shared = rand_layer(rng, T, d, m, E, k, ms, bf16=False)
    dy = rng.standard_normal((T, d))
    y, saved = om.forward(x, logits, experts, k, "fp64", shared=shared)
    gr = om.backward(dy, x, experts, k, "fp64", saved, shared=shared)
    eps = 1e-6

    def fd(f, a, i):
        a[i] += eps
        lp = f()
        a[i] -= 2 * eps
        lm = f()
        a[i] += eps
        return (lp - lm) / (2 * eps)

    L = lambda: _loss(x, logits, experts, k, shared, dy)
    for i in [(0, 0), (3, 5), (6, 7)]:
        assert np.isclose(fd(L, x, i), gr["dx"][i], rtol=1e-6, atol=1e-8)
    for e in range(E):
        if e not in gr["dW_gu"]:
            continue
        for i in [(0, 0), (5, 3), (7, 7)]:
            assert np.isclose(fd(L, experts[e][0], i), gr["dW_gu"][e][i], rtol=1e-6, atol=1e-8)
        for i in [(0, 0), (7, 3)]:
            assert np.isclose(fd(L, experts[e][1], i), gr["dW_dn"][e][i], rtol=1e-6, atol=1e-8)
    for i in [(1, 2), (6, 0)]:
        assert np.isclose(fd(L, shared[0], i), gr["dWs_gu"][i], rtol=1e-6, atol=1e-8)
        assert np.isclose(fd(L, shared[1], (i[1], i[0] % ms)), gr["dWs_dn"][i[1], i[0] % ms], rtol=1e-6, atol=1e-8)
    # logits: perturb only entries whose perturbation cannot change the top-k set
    lg = logits.astype(np.float64)
    checked = 0
    for t in range(T):
        srt = np.sort(lg[t])[::-1]
        if srt[k - 1] - srt[k] < 1e-3:
            continue
        for e in range(E):
            lp = lg.copy(); lp[t, e] += 1e-4
            lm = lg.copy(); lm[t, e] -= 1e-4
            num = (_loss(x, lp.astype(np.float32), experts, k, shared, dy)
                   - _loss(x, lm.astype(np.float32), experts, k, shared, dy))
            dl = np.float32(lg[t, e] + 1e-4).astype(np.float64) - np.float32(lg[t, e] - 1e-4).astype(np.float64)
            assert np.isclose(num / dl, gr["dlogits"][t, e], rtol=1e-3, atol=1e-6)
            checked += 1
    assert checked >= E * 3
    # unselected experts get exactly zero
    mask = np.zeros((T, E), bool)
    np.put_along_axis(mask, saved["idx"], True, 1)
    assert np.all(gr["dlogits"][~mask] == 0)


def test_dlogits_closed_form_sums_to_zero():
    rng = np.random.default_rng(13)
    x, logits, experts, _ = rand_layer(rng, 30, 16, 8, 6, 3)
    dy = nx.bf16_round(rng.standard_normal((30, 16)))
    _, saved = om.forward(x, logits, experts, 3, "bf16")
    gr = om.backward(dy, x, experts, 3, "bf16", saved)
    assert np.allclose(gr["dlogits"].sum(1), 0.0, atol=1e-12)   # softmax gradient is orthogonal to 1


@pytest.mark.parametrize("fmt,tol", [("bf16", 3e-2), ("mxfp8", 1e-1)])
def test_backward_rounded_formats_close_to_exact(fmt, tol):
    rng = np.random.default_rng(14)
    T, d, m, E, k, ms = 50, 64, 32, 4, 2, 32
    x, logits, experts, shared = rand_layer(rng, T, d, m, E, k, ms)
    dy = nx.bf16_round(rng.standard_normal((T, d)))
    _, s64 = om.forward(x, logits, experts, k, "fp64", shared=shared)
    g64 = om.backward(dy, x, experts, k, "fp64", s64, shared=shared)
    _, s = om.forward(x, logits, experts, k, fmt, shared=shared)
    g = om.backward(dy, x, experts, k, fmt, s, shared=shared)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(g["dx"], g64["dx"]) < tol
    assert rel(g["dlogits"], g64["dlogits"]) < tol
    for e in g64["dW_gu"]:
        assert rel(g["dW_gu"][e], g64["dW_gu"][e]) < tol
        assert rel(g["dW_dn"][e], g64["dW_dn"][e]) < tol
    assert rel(g["dWs_gu"], g64["dWs_gu"]) < tol


def test_column_blocks_start_at_first_row_and_pad_at_end():
    """Column blocks are rows [0, 32), [32, 64), ... of the expert, the last one
    zero-padded: rows 0..31 scaled by 2**8 and rows 32..44 by 2**-8 are exact
    in those blocks, while any block straddling row 32 (padding in front, or
    blocks counted from the last row) mixes scales 16 binades apart and loses
    bits."""
    rng = np.random.default_rng(15)
    a = _mant(rng, (45, 32)) * 2.0 ** rng.integers(-2, 3, (1, 32))
    a[:32] *= 2.0 ** 8
    a[32:] *= 2.0 ** -8
    assert np.array_equal(om._col_blocks(a), a)
    front = np.concatenate([np.zeros((19, 32)), a])
    assert not np.array_equal(nx.mx_roundtrip(front, axis=0)[19:], a)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8"])
def test_prepared_operands_change_nothing(fmt):
    """Weight preparation (S0) done ahead of time gives bit-identical results."""
    rng = np.random.default_rng(16)
    T, d, m, E, k = 37, 64, 32, 4, 2
    x, logits, experts, _ = rand_layer(rng, T, d, m, E, k)
    dy = nx.bf16_round(rng.standard_normal((T, d)))
    prepped = [(g, n, om.prepare_expert(g, n, fmt)) for g, n in experts]
    y1, s1 = om.forward(x, logits, experts, k, fmt)
    y2, s2 = om.forward(x, logits, prepped, k, fmt)
    assert np.array_equal(y1, y2)
    g1 = om.backward(dy, x, experts, k, fmt, s1)
    g2 = om.backward(dy, x, prepped, k, fmt, s2)
    for key in ("dx", "dlogits"):
        assert np.array_equal(g1[key], g2[key])
    for e in g1["dW_gu"]:
        assert np.array_equal(g1["dW_gu"][e], g2["dW_gu"][e]) and np.array_equal(g1["dW_dn"][e], g2["dW_dn"][e])


# ---------------------------------------------------------------- MXFP8 quantisation axes
# Each test below builds operands that are exactly representable in MXFP8 along
# the axis the reading names (blocks of 32 along the GEMM's K for dgrad and the
# forward; blocks of 32 rows of one expert for wgrad) and wildly scaled along
# the other axis, so the quantised products equal the unquantised float64 ones
# exactly, while quantising along the other axis would lose bits.  The
# "wrong axis is lossy" premise of every operand is asserted too.
def _mant(rng, shape):
    """Signed values with 3 fraction bits in [1, 1.75]: E4M3 mantissas that
    never saturate at the top of a block."""
    return (rng.integers(8, 15, shape) * rng.choice([-1, 1], shape)) / 8.0


def _row_exact(a):
    return np.array_equal(nx.mx_roundtrip(a, axis=1), a)


def _col_exact(a):
    return np.array_equal(om._col_blocks(a), a)


def test_mx_h_quantised_along_m():
    """Forward: h is quantised along m (its GEMM's K) straight from the SwiGLU
    output.  G = 64 everywhere makes silu(G) = G exactly in float64 (exp(-64)
    vanishes against 1), and U = X[:, 1:m+1], so h = 64 * X[:, 1:m+1]: rows of
    one binade range each, rows 2**-9 .. 2**9 apart."""
    rng = np.random.default_rng(31)
    n, d, m = 64, 64, 32
    X = np.zeros((n, d))
    X[:, 0] = 1.0
    X[:, 1:m + 1] = _mant(rng, (n, m)) * 2.0 ** rng.integers(-9, 10, (n, 1))
    W_gu = np.zeros((2 * m, d))
    W_gu[:m, 0] = 64.0                                  # gate: G = 64 * x[:, 0]
    W_gu[m + np.arange(m), 1 + np.arange(m)] = 1.0      # up: U = X[:, 1:m+1]
    W_dn = _mant(rng, (d, m)) * 2.0 ** rng.integers(-2, 3, (d, 1))
    h = 64.0 * X[:, 1:m + 1]
    assert _row_exact(X) and _row_exact(W_gu) and _row_exact(W_dn)
    assert _row_exact(h) and not _col_exact(h)
    res = om.expert_forward(X, W_gu, W_dn, "mxfp8")
    assert np.array_equal(res["G"], np.full((n, m), 64.0)) and np.array_equal(res["U"], X[:, 1:m + 1])
    assert np.array_equal(res["o"], nx.bf16_round(h @ W_dn.T))


def _bwd_ops(dn_bwd, gu_bwd):
    return dict(gu_fwd=None, dn_fwd=None, dn_bwd=dn_bwd, gu_bwd=gu_bwd)


def test_mx_dgrad_operands_quantised_along_k():
    """Backward dgrads: dO is quantised along d (the down dgrad's K) and dGU
    along 2m (the gate/up dgrad's K).  dO rows are 2**-9 .. 2**9 apart; the
    down weight copy W_dn^T = [I | 0] makes dh = dO[:, :m]; G = 0 makes the
    SwiGLU backward dG = dh * U / 2 (silu'(0) = 1/2) and dU = 0 (silu(0) = 0),
    with U = 2**b per row, so dGU keeps dO's per-row scales."""
    rng = np.random.default_rng(32)
    n, d, m = 64, 64, 32
    dO = _mant(rng, (n, d)) * 2.0 ** rng.integers(-9, 10, (n, 1))
    U = np.broadcast_to(2.0 ** rng.integers(-4, 5, (n, 1)), (n, m))
    GU = np.concatenate([np.zeros((n, m)), U], axis=1)
    dn_bwd = np.eye(m, d)
    gu_bwd = _mant(rng, (d, 2 * m)) * 2.0 ** rng.integers(-1, 2, (d, 1))
    dGU = np.concatenate([dO[:, :m] * U / 2.0, np.zeros((n, m))], axis=1)
    assert _row_exact(dO) and not _col_exact(dO)
    assert _row_exact(dGU) and not _col_exact(dGU)
    X = nx.bf16_round(rng.standard_normal((n, d)))
    h = nx.bf16_round(rng.standard_normal((n, m)))
    res = om.expert_backward(dO, X, GU, h, np.zeros((2 * m, d)), np.zeros((d, m)), "mxfp8",
                             _bwd_ops(dn_bwd, gu_bwd))
    assert np.array_equal(res["dh"], dO[:, :m])
    assert np.array_equal(res["dGU"], dGU)
    assert np.array_equal(res["dX"], nx.bf16_round(dGU @ gu_bwd.T))


def test_mx_wgrad_operands_quantised_in_column_blocks():
    """Backward wgrads: dO, h, dGU and X are quantised in blocks of 32
    consecutive rows of the expert (the wgrad's K), the last block zero-padded
    (n = 50: blocks of 32 and 18 rows).  Columns are 2**-9 .. 2**9 apart; the
    first m columns of dO (which feed dh through W_dn^T = [I | 0]) stay within
    a 3-binade range per row so that dh = dO[:, :m] exactly, and U = 2**u per
    column gives dG = dh * U / 2 per-column scales.  Rows 0..31 carry an extra
    2**9 and rows 32..49 2**-9, so blocks that do not start at rows 0 and 32
    would mix scales 18 binades apart."""
    rng = np.random.default_rng(33)
    n, d, m = 50, 64, 32
    blk = np.where(np.arange(n) < 32, 2.0 ** 9, 2.0 ** -9)[:, None]
    dO = _mant(rng, (n, d)) * 2.0 ** rng.integers(-9, 10, (1, d)) * blk
    dO[:, :m] = _mant(rng, (n, m)) * 2.0 ** rng.integers(-1, 2, (n, 1)) * blk
    h = _mant(rng, (n, m)) * 2.0 ** rng.integers(-9, 10, (1, m)) * blk
    X = _mant(rng, (n, d)) * 2.0 ** rng.integers(-9, 10, (1, d)) * blk
    U = np.broadcast_to(2.0 ** rng.integers(-9, 10, (1, m)), (n, m))
    GU = np.concatenate([np.zeros((n, m)), U], axis=1)
    dGU = np.concatenate([dO[:, :m] * U / 2.0, np.zeros((n, m))], axis=1)
    for a in (dO, h, X, dGU):
        assert _col_exact(a) and not _row_exact(a)
        shifted = np.concatenate([np.zeros((14, a.shape[1])), a])       # blocks counted from the end
        assert not np.array_equal(nx.mx_roundtrip(shifted, axis=0)[14:], a)
    assert _row_exact(dO[:, :m])
    res = om.expert_backward(dO, X, GU, h, np.zeros((2 * m, d)), np.zeros((d, m)), "mxfp8",
                             _bwd_ops(np.eye(m, d), np.zeros((d, 2 * m))))
    assert np.array_equal(res["dGU"], dGU)
    assert np.array_equal(res["dW_dn"], nx.bf16_round(dO.T @ h))
    assert np.array_equal(res["dW_gu"], nx.bf16_round(dGU.T @ X))
