"""Router projection in front of the layer and the load-balancing term, in
float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages make token routing the first stage fused into the layer
(daily-ai-frontier summary, TL;DR) but define neither the router projection
nor a balancing term.  Readings (each one is also listed in the design notes
of the repository):

* router: logits = x W_r^T, a bias-free linear projection of bfloat16 tokens
  x [T, d] by bfloat16 router weights W_r [E, d]; float64 here, fp32
  accumulation and fp32 logits on the device;
* load balancing: the auxiliary loss of the Switch Transformer, taken over
  the k routed slots of every token,
      L = alpha * E * sum_e f_e * P_e,
      f_e = counts_e / (T * k)                (fraction of slots on expert e),
      P_e = (1 / T) * sum_t softmax(logits_t)_e   (over all E experts);
  f is piecewise constant in the logits, so the gradient flows through P only:
      dL/dl[t, j] = alpha * E / T * p[t, j] * (f_j - sum_e f_e p[t, e]);
  the loss enters the training objective with weight 1;
* router backward: dlogits (the layer's plus the loss's) is rounded to
  bfloat16; dx_total = bf16(dx + dlogits W_r) (one rounding of the sum) and
  dW_r = bf16(dlogits^T x).
"""
import numpy as np

from .numerics import bf16_round


def router_logits(x, W_r):
    """logits [T, E] = x [T, d] @ W_r [E, d]^T."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(W_r, dtype=np.float64).T


def softmax_full(logits):
    """Row softmax over all E experts."""
    l64 = np.asarray(logits, dtype=np.float64)
    ex = np.exp(l64 - l64.max(axis=1, keepdims=True))
    return ex / ex.sum(axis=1, keepdims=True)


def balance_terms(logits, counts, k):
    """(f [E], P [E], p [T, E]) of the load-balancing loss."""
    p = softmax_full(logits)
    T = p.shape[0]
    f = np.asarray(counts, dtype=np.float64) / (T * k)
    P = p.mean(axis=0)
    return f, P, p


def aux_loss(logits, counts, k, alpha):
    """Load-balancing loss and its gradient with respect to the logits
    (counts held fixed: they are piecewise constant in the logits)."""
    f, P, p = balance_terms(logits, counts, k)
    T, E = p.shape
    loss = alpha * E * float(np.dot(f, P))
    s = p @ f                                   # sum_e f_e p[t, e], per token
    grad = alpha * E / T * p * (f[None, :] - s[:, None])
    return loss, grad


def router_backward(dlogits, x, W_r, dx, fmt="bf16"):
    """(dx_total, dW_r) of the router projection.  fmt "fp64" skips every
    rounding (used by the finite-difference pins)."""
    rnd = (lambda a: a) if fmt == "fp64" else bf16_round
    g = rnd(np.asarray(dlogits, dtype=np.float64))
    dx_total = rnd(np.asarray(dx, dtype=np.float64) + g @ np.asarray(W_r, dtype=np.float64))
    dW_r = rnd(g.T @ np.asarray(x, dtype=np.float64))
    return dx_total, dW_r
