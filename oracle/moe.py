"""The mixture-of-experts layer, step by step, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Notation: T tokens, d hidden, m expert intermediate, E experts, k experts per
token, R = T*k routed rows.  Flat slot i = t*k + j is the j-th expert choice
of token t.  Expert-sorted row r is the position of a slot after a stable
sort of all slots by expert.

Steps, in the pages' order (the "Mixture-of-Kittens" wiki page, flowchart and
Key claims; the aiexpert.news article):

1. route     -- top-k expert choice per token and its combine weights
                (token routing is the first stage fused into the layer:
                daily-ai-frontier summary, TL;DR).
2. schedule  -- per-expert counts, exclusive offsets and the token
                permutation, all computed on the device with no host sync
                (wiki page, flowchart "device-side schedule kernel" and Key
                claims "CPU-free scheduling").
3. dispatch  -- rows gathered into expert-contiguous order, MXFP8
                quantisation of activations fused in (Key claims, MXFP8
                bullet).
4. experts   -- grouped GEMMs: gate/up, SwiGLU, quantisation, down (flowchart
                "Expert grouped GEMMs, MXFP8 + fused SwiGLU + fused
                quantization").
5. combine   -- weighted sum of each token's k expert outputs in a fixed
                order, so the result is bitwise reproducible (wiki page,
                TL;DR last paragraph and Key claims "Bitwise determinism").
6. shared    -- an always-on BF16 shared expert (Key claims, MXFP8 bullet:
                "the shared expert stays BF16").
7. backward  -- reverse-combine then reverse-dispatch (Key claims,
                communication-direction bullet); the formulas are the chain
                rule of steps 1-6.

Readings where the pages are silent (each one is also listed in the design
notes of the repository):

* top-k is taken on the raw fp32 logits, ties broken by the lower expert
  index; softmax over all E followed by renormalisation over the chosen k is
  identical to a softmax over the chosen k, which is what is computed;
* rows of one expert keep ascending flat-slot order (stable sort);
* the gate half is the first m rows of W_gu[e] ([2m, d]); h = silu(G) * U;
* every GEMM output that is stored (o, s, dX, dW, ...) is rounded to
  bfloat16 once; h is rounded to bfloat16 on the BF16 path and MX-quantised
  straight from the unrounded SwiGLU output on the MXFP8 path;
* the combine adds slots j = 0..k-1 in order, then the shared expert, and
  rounds once;
* backward: gradients pass straight through the quantisers; dO = w*dy and
  dGU are materialised in bfloat16 and every MXFP8 backward operand is
  quantised from bfloat16 values: row blocks (32 along the GEMM's K) for
  dgrad, column blocks (32 consecutive rows of one expert, zero-padded) for
  wgrad; the forward saves G, U and h in bfloat16.
"""
import numpy as np

from .numerics import bf16_round, mx_roundtrip, MX_BLOCK
from .nvfp4 import global_scale, nvfp4_roundtrip

FORMATS = ("bf16", "mxfp8", "nvfp4", "fp64")


def _rnd(fmt):
    return (lambda a: a) if fmt == "fp64" else bf16_round


def sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


# ----------------------------------------------------------------------------
# 1. route
# ----------------------------------------------------------------------------
def route(logits, k):
    """Top-k experts per token and their combine weights.

    Experts are ordered by (logit descending, index ascending) and the first
    k are kept; slot j holds the j-th.  The weights are the softmax over the
    k chosen logits, w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), in float64.
    Returns idx [T, k] int64 and w [T, k] float64.
    """
    logits = np.asarray(logits)
    assert logits.dtype == np.float32, "router logits are fp32"
    l64 = logits.astype(np.float64)
    order = np.argsort(-l64, axis=1, kind="stable")   # stable: equal logits keep lower index first
    idx = order[:, :k].astype(np.int64)
    sel = np.take_along_axis(l64, idx, axis=1)
    ex = np.exp(sel - sel[:, :1])
    w = ex / ex.sum(axis=1, keepdims=True)
    return idx, w


# ----------------------------------------------------------------------------
# 2. schedule
# ----------------------------------------------------------------------------
def schedule(idx, E):
    """Per-expert counts, exclusive offsets, and the stable permutation.

    counts[e] = number of slots routed to e; offsets = exclusive prefix sum
    (length E+1, offsets[E] = R); perm[i] = expert-sorted row of flat slot i;
    inv[r] = flat slot at row r (inv is perm's inverse).
    """
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    inv = np.argsort(flat, kind="stable").astype(np.int64)
    perm = np.empty_like(inv)
    perm[inv] = np.arange(flat.size, dtype=np.int64)
    return counts, offsets, perm, inv


# ----------------------------------------------------------------------------
# 0. weight preparation (S0)
# ----------------------------------------------------------------------------
def prepare_expert(W_gu, W_dn, fmt, backward=True, forward=True):
    """Operands the expert GEMMs read, from the bf16 masters of one expert.

    MXFP8 is the default expert format ("Mixture-of-Kittens" wiki page, Key
    claims, MXFP8 bullet): the forward operands are W_gu [2m, d] and W_dn
    [d, m] quantised along their K (d, m); the backward dgrad operands are
    W_dn^T [m, d] quantised along d and W_gu^T [d, 2m] quantised along 2m.
    NVFP4 (forward only; the NVFP4 variant of the expert GEMMs): each
    expert matrix is one tensor with its own second-level scale, quantised in
    blocks of 16 along K.  Values are returned dequantised (float64).  Other
    formats use the masters.  ``forward`` / ``backward`` select which of the
    two pairs are made.
    """
    W_gu = np.asarray(W_gu, dtype=np.float64)
    W_dn = np.asarray(W_dn, dtype=np.float64)
    ops = {}
    if fmt == "nvfp4":
        if backward:
            raise NotImplementedError("the NVFP4 variant is forward only")
        if forward:
            ops["gu_fwd"] = nvfp4_roundtrip(W_gu, global_scale(np.abs(W_gu).max()), axis=1)
            ops["dn_fwd"] = nvfp4_roundtrip(W_dn, global_scale(np.abs(W_dn).max()), axis=1)
    elif fmt == "mxfp8":
        if forward:
            ops["gu_fwd"] = mx_roundtrip(W_gu, axis=1)
            ops["dn_fwd"] = mx_roundtrip(W_dn, axis=1)
        if backward:
            ops["dn_bwd"] = mx_roundtrip(W_dn.T, axis=1)
            ops["gu_bwd"] = mx_roundtrip(W_gu.T, axis=1)
    else:
        if forward:
            ops.update(gu_fwd=W_gu, dn_fwd=W_dn)
        if backward:
            ops.update(dn_bwd=W_dn.T, gu_bwd=W_gu.T)
    return ops


def _unpack(item):
    """experts[e] is (W_gu, W_dn) or (W_gu, W_dn, prepared operands)."""
    return (item[0], item[1], item[2]) if len(item) == 3 else (item[0], item[1], None)


# ----------------------------------------------------------------------------
# 3./4. one expert
# ----------------------------------------------------------------------------
def _col_blocks(a):
    """MX round trip of ``a`` [n, c] in blocks of 32 rows (zero-padded at the end)."""
    n = a.shape[0]
    pad = (-n) % MX_BLOCK
    ap = np.concatenate([a, np.zeros((pad,) + a.shape[1:])], axis=0) if pad else a
    return mx_roundtrip(ap, axis=0)[:n]


def expert_forward(X, W_gu, W_dn, fmt, ops=None, x_scale=None):
    """SwiGLU FFN of one expert on its gathered rows.

    X [n, d] bf16 values; W_gu [2m, d] (gate rows first); W_dn [d, m].
    MXFP8: X, W_gu and W_dn are quantised along K (d, d, m); h is
    quantised along m straight from the float64 SwiGLU output.
    NVFP4: the same axes in blocks of 16; X with the second-level scale
    ``x_scale`` of the layer's whole x (from X itself when not given), h
    rounded to fp32 and quantised with second-level scale 1.
    ``ops`` are the expert's prepared operands (:func:`prepare_expert`),
    computed here when not given.
    Returns dict(G, U (unrounded), GU_saved [n, 2m], h_saved [n, m], o [n, d]).
    """
    m = W_gu.shape[0] // 2
    rnd = _rnd(fmt)
    if ops is None:
        ops = prepare_expert(W_gu, W_dn, fmt, backward=False)
    if fmt == "mxfp8":
        Xq = mx_roundtrip(X, axis=1)
    elif fmt == "nvfp4":
        Xq = nvfp4_roundtrip(X, global_scale(np.abs(X).max()) if x_scale is None else x_scale, axis=1)
    else:
        Xq = X
    Wq, Dq = ops["gu_fwd"], ops["dn_fwd"]
    G = Xq @ Wq[:m].T
    U = Xq @ Wq[m:].T
    h = silu(G) * U
    if fmt == "mxfp8":
        h_op = mx_roundtrip(h, axis=1)
    elif fmt == "nvfp4":
        h_op = nvfp4_roundtrip(h.astype(np.float32).astype(np.float64), 1.0, axis=1)
    else:
        h_op = rnd(h)
    o = rnd(h_op @ Dq.T)
    return dict(G=G, U=U, GU_saved=rnd(np.concatenate([G, U], axis=1)), h_saved=rnd(h), o=o)


def shared_forward(x, Ws_gu, Ws_dn, fmt):
    """Always-on BF16 shared SwiGLU expert (fp64 format: no rounding)."""
    sfmt = "fp64" if fmt == "fp64" else "bf16"
    return expert_forward(x, Ws_gu, Ws_dn, sfmt)


# ----------------------------------------------------------------------------
# full forward
# ----------------------------------------------------------------------------
def forward(x, logits, experts, k, fmt, shared=None, x_scale=None):
    """Layer forward.

    x [T, d] (bf16 values as float64); logits [T, E] fp32; ``experts[e]``
    returns (W_gu [2m, d], W_dn [d, m]) float64 and ``len(experts)`` is E;
    ``shared`` is None or (Ws_gu [2m_s, d], Ws_dn [d, m_s]).
    NVFP4: ``x_scale`` is the second-level scale of x (computed from x when
    not given; a caller passing a subset of the tokens passes the whole x's).
    Returns (y [T, d], saved dict).
    """
    assert fmt in FORMATS
    x = np.asarray(x, dtype=np.float64)
    if fmt == "nvfp4" and x_scale is None:
        x_scale = global_scale(np.abs(x).max())
    T, d = x.shape
    E = len(experts)
    R = T * k
    rnd = _rnd(fmt)
    idx, w = route(logits, k)
    counts, offsets, perm, inv = schedule(idx, E)
    row_tok = inv // k
    o = np.zeros((R, d))
    GU = None
    h_saved = None
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        W_gu, W_dn, ops = _unpack(experts[e])
        res = expert_forward(x[row_tok[r0:r1]], W_gu, W_dn, fmt, ops, x_scale=x_scale)
        if GU is None:
            m = W_gu.shape[0] // 2
            GU = np.zeros((R, 2 * m))
            h_saved = np.zeros((R, m))
        o[r0:r1] = res["o"]
        GU[r0:r1] = res["GU_saved"]
        h_saved[r0:r1] = res["h_saved"]
    s = None
    sres = None
    if shared is not None:
        sres = shared_forward(x, shared[0], shared[1], fmt)
        s = sres["o"]
    acc = np.zeros((T, d))
    for j in range(k):                              # fixed slot order
        acc = acc + w[:, j:j + 1] * o[perm.reshape(T, k)[:, j]]
    if s is not None:
        acc = acc + s
    y = rnd(acc)
    saved = dict(idx=idx, w=w, counts=counts, offsets=offsets, perm=perm, inv=inv,
                 o=o, GU=GU, h=h_saved, s=s, shared=sres)
    return y, saved


# ----------------------------------------------------------------------------
# 7. backward
# ----------------------------------------------------------------------------
def swiglu_backward(dh, G, U):
    """dG = dh * U * silu'(G), dU = dh * silu(G), silu'(g) = s(1 + g(1 - s)), s = sigmoid(g)."""
    s = sigmoid(G)
    dG = dh * U * s * (1.0 + G * (1.0 - s))
    dU = dh * G * s
    return dG, dU


def expert_backward(dO, X, GU, h, W_gu, W_dn, fmt, ops=None):
    """Backward of one expert on its rows.

    dO [n, d] bf16 values (w * dy), X [n, d], GU [n, 2m] and h [n, m] saved
    in bf16.  Returns dict(dX [n, d], dW_gu [2m, d], dW_dn [d, m]).
    MXFP8: dgrad operands are quantised in blocks of 32 along the GEMM's K
    (dO along d, dGU along 2m, the weight copies W_dn^T along d and W_gu^T
    along 2m); wgrad operands in blocks of 32 rows (dO, h, dGU, X).
    """
    m = W_gu.shape[0] // 2
    rnd = _rnd(fmt)
    if ops is None or "dn_bwd" not in ops:
        ops = prepare_expert(W_gu, W_dn, fmt, backward=True)
    G, U = GU[:, :m], GU[:, m:]
    if fmt == "mxfp8":
        dh = mx_roundtrip(dO, axis=1) @ ops["dn_bwd"].T
    else:
        dh = dO @ ops["dn_bwd"].T
    dG, dU = swiglu_backward(dh, G, U)
    dGU = rnd(np.concatenate([dG, dU], axis=1))
    if fmt == "mxfp8":
        dW_dn = _col_blocks(dO).T @ _col_blocks(h)
        dX = mx_roundtrip(dGU, axis=1) @ ops["gu_bwd"].T
        dW_gu = _col_blocks(dGU).T @ _col_blocks(X)
    else:
        dW_dn = dO.T @ h
        dX = dGU @ ops["gu_bwd"].T
        dW_gu = dGU.T @ X
    return dict(dX=rnd(dX), dW_gu=rnd(dW_gu), dW_dn=rnd(dW_dn), dGU=dGU, dh=dh)


def shared_backward(dy, x, sres, Ws_gu, Ws_dn, fmt):
    """BF16 shared expert backward: its output gradient is dy itself."""
    sfmt = "fp64" if fmt == "fp64" else "bf16"
    return expert_backward(dy, x, sres["GU_saved"], sres["h_saved"], Ws_gu, Ws_dn, sfmt)


def backward(dy, x, experts, k, fmt, saved, shared=None, dw_experts=None):
    """Layer backward.

    dy [T, d] bf16 values.  Returns dict(dx [T, d], dlogits [T, E] fp64,
    dW_gu {e: [2m, d]}, dW_dn {e: [d, m]}, dWs_gu, dWs_dn, and the
    expert-sorted intermediates dO [R, d], dX [R, d], dGU [R, 2m], g [T, k]).  ``dw_experts``
    restricts which experts get weight gradients (all when None); dx and
    dlogits always cover every token.
    """
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    T, d = x.shape
    E = len(experts)
    rnd = _rnd(fmt)
    idx, w, offsets, perm, inv = (saved[n] for n in ("idx", "w", "offsets", "perm", "inv"))
    row_tok = inv // k
    row_j = inv % k
    row_w = w[row_tok, row_j]
    R = T * k
    # B1 reverse-combine: dO rows and g = <dy, o> per slot
    dO = rnd(row_w[:, None] * dy[row_tok])
    g_rows = np.einsum("rc,rc->r", dy[row_tok], saved["o"])
    g = g_rows[perm].reshape(T, k)
    # B2-B5 per expert
    dX = np.zeros((R, d))
    dGU = None
    dW_gu, dW_dn = {}, {}
    want = set(range(E)) if dw_experts is None else set(dw_experts)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            if e in want:
                W_gu, W_dn, _ = _unpack(experts[e])
                dW_gu[e] = np.zeros_like(W_gu)
                dW_dn[e] = np.zeros_like(W_dn)
            continue
        W_gu, W_dn, ops = _unpack(experts[e])
        res = expert_backward(dO[r0:r1], x[row_tok[r0:r1]], saved["GU"][r0:r1],
                              saved["h"][r0:r1], W_gu, W_dn, fmt, ops)
        dX[r0:r1] = res["dX"]
        if dGU is None:
            dGU = np.zeros((R, res["dGU"].shape[1]))
        dGU[r0:r1] = res["dGU"]
        if e in want:
            dW_gu[e] = res["dW_gu"]
            dW_dn[e] = res["dW_dn"]
    # B7 shared expert
    dxs = None
    dWs_gu = dWs_dn = None
    if shared is not None:
        sb = shared_backward(dy, x, saved["shared"], shared[0], shared[1], fmt)
        dxs, dWs_gu, dWs_dn = sb["dX"], sb["dW_gu"], sb["dW_dn"]
    # B6 reverse-dispatch: fixed slot order, then the shared expert, one rounding
    acc = np.zeros((T, d))
    for j in range(k):
        acc = acc + dX[perm.reshape(T, k)[:, j]]
    if dxs is not None:
        acc = acc + dxs
    dx = rnd(acc)
    # dlogits: softmax over the chosen k, closed form w_j (g_j - sum_i w_i g_i)
    dl_sel = w * (g - (w * g).sum(axis=1, keepdims=True))
    dlogits = np.zeros((T, E))
    np.put_along_axis(dlogits, idx, dl_sel, axis=1)
    return dict(dx=dx, dlogits=dlogits, dW_gu=dW_gu, dW_dn=dW_dn, dWs_gu=dWs_gu,
                dWs_dn=dWs_dn, dO=dO, g=g, dX=dX, dGU=dGU)


# ----------------------------------------------------------------------------
# weight quantisation (S0)
# ----------------------------------------------------------------------------
def quantize_weights(W, transpose=False):
    """MXFP8 codes and scale bytes of weight matrices W [..., rows, cols].

    transpose=False quantises along cols (the forward K); transpose=True
    returns the quantisation of W^T (per matrix) along its last axis, i.e.
    blocks of 32 along the original rows (the backward copies).
    """
    from .numerics import mx_quantize
    W = np.asarray(W, dtype=np.float64)
    if transpose:
        W = np.swapaxes(W, -1, -2)
    return mx_quantize(W, axis=-1)
