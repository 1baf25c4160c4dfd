"""Pins of the router / load-balancing oracle against special cases, closed
forms and finite differences (CPU only)."""
import numpy as np

from oracle import router as orr


def test_router_logits_one_hot_tokens_pick_weight_columns():
    # x row t = unit vector e_{j(t)}: logits[t] = W_r[:, j(t)] (catches a transposed operand)
    rng = np.random.default_rng(0)
    E, d, T = 6, 10, 7
    W = rng.standard_normal((E, d))
    j = rng.integers(0, d, T)
    x = np.zeros((T, d))
    x[np.arange(T), j] = 1.0
    assert np.array_equal(orr.router_logits(x, W), W[:, j].T)


def test_aux_loss_uniform_router_balanced_load_is_alpha_with_zero_gradient():
    T, E, k, alpha = 64, 8, 2, 0.01
    logits = np.zeros((T, E), dtype=np.float32)
    counts = np.full(E, T * k // E)
    loss, grad = orr.aux_loss(logits, counts, k, alpha)
    assert abs(loss - alpha) < 1e-15
    assert np.abs(grad).max() < 1e-18


def test_aux_loss_all_slots_on_one_expert():
    # f = e_0, so L = alpha * E * P_0 with P_0 the mean probability of expert 0
    rng = np.random.default_rng(1)
    T, E, k, alpha = 50, 5, 1, 0.3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    counts = np.zeros(E)
    counts[0] = T * k
    loss, _ = orr.aux_loss(logits, counts, k, alpha)
    l = logits.astype(np.float64)
    p0 = np.exp(l[:, 0]) / np.exp(l).sum(axis=1)
    assert abs(loss - alpha * E * p0.mean()) < 1e-14


def test_aux_loss_gradient_matches_central_differences():
    rng = np.random.default_rng(2)
    T, E, k, alpha = 9, 6, 2, 0.7
    logits = rng.standard_normal((T, E))
    counts = rng.integers(0, 10, E)
    _, grad = orr.aux_loss(logits, counts, k, alpha)
    h = 1e-6
    num = np.zeros_like(logits)
    for t in range(T):
        for e in range(E):
            lp, lm = logits.copy(), logits.copy()
            lp[t, e] += h
            lm[t, e] -= h
            num[t, e] = (orr.aux_loss(lp, counts, k, alpha)[0] - orr.aux_loss(lm, counts, k, alpha)[0]) / (2 * h)
    assert np.abs(num - grad).max() < 1e-8


def test_router_backward_matches_central_differences():
    # S(x, W) = <G, x W^T>: dS/dx = G W, dS/dW = G^T x (fp64, no rounding)
    rng = np.random.default_rng(3)
    T, E, d = 4, 3, 5
    x, W, G = rng.standard_normal((T, d)), rng.standard_normal((E, d)), rng.standard_normal((T, E))
    dx0 = rng.standard_normal((T, d))
    dx_total, dW = orr.router_backward(G, x, W, dx0, fmt="fp64")

    def S(xv, Wv):
        return float((G * orr.router_logits(xv, Wv)).sum())

    h = 1e-6
    num_x = np.zeros_like(x)
    for i in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        num_x[i] = (S(xp, W) - S(xm, W)) / (2 * h)
    num_W = np.zeros_like(W)
    for i in np.ndindex(W.shape):
        Wp, Wm = W.copy(), W.copy()
        Wp[i] += h
        Wm[i] -= h
        num_W[i] = (S(x, Wp) - S(x, Wm)) / (2 * h)
    assert np.abs((dx_total - dx0) - num_x).max() < 1e-7
    assert np.abs(dW - num_W).max() < 1e-7


def test_router_backward_rounds_once():
    # bf16 path: dlogits rounded to bf16, the sum dx + dlogits W rounded once
    from oracle.numerics import bf16_round
    rng = np.random.default_rng(4)
    T, E, d = 3, 4, 6
    x = bf16_round(rng.standard_normal((T, d)))
    W = bf16_round(rng.standard_normal((E, d)))
    G = rng.standard_normal((T, E))
    dx0 = bf16_round(rng.standard_normal((T, d)))
    dx_total, dW = orr.router_backward(G, x, W, dx0)
    g = bf16_round(G)
    assert np.array_equal(dx_total, bf16_round(dx0 + g @ W))
    assert np.array_equal(bf16_round(dx_total), dx_total)
    assert np.array_equal(dW, bf16_round(g.T @ x))
