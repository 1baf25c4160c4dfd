"""A torch drop-in for the MoE layer: an autograd.Function around the C ABI
and an nn.Module that owns the bf16 master weights as parameters.

Every computation runs in the library's kernels; this file only moves
pointers.  The forward re-derives the kernels' weight operands (MXFP8 codes in
both orientations, or bf16 transposes) from the current masters, so an
optimizer step on the parameters is seen by the next forward; its cost is the
weight preparation step of a training update.  Gradients pass straight through
the MXFP8 quantisers, so the masters receive the gradients the library
computes for the quantised layer.  Each training forward keeps its activations
in its own buffer, so several forwards may precede their backwards.
"""
import torch

from .layer import MoELayer


class MoEFunction(torch.autograd.Function):
    """y = moe(x, logits; W_gu, W_dn[, Ws_gu, Ws_dn]) for the shapes of `layer`.

    x [T, d] bf16, logits [T, E] fp32 -> y [T, d] bf16.  With router weights
    W_r [E, d] (bf16) the logits are computed from x instead (pass logits =
    None); the router's backward then adds its dx contribution in place and
    returns dW_r.  Backward returns dx, dlogits (fp32; with a load-balancing
    term its gradient is included) and the gradients of the bf16 weights."""

    @staticmethod
    def forward(ctx, x, logits, W_r, W_gu, W_dn, Ws_gu, Ws_dn, layer):
        layer.prepare_from(W_gu, W_dn, Ws_gu, Ws_dn)
        x = x.contiguous()
        if W_r is not None:
            logits = layer.router_logits(x, W_r.contiguous())
        need = any(ctx.needs_input_grad[:7])
        saved = layer.new_saved() if need else None
        y = layer.forward(x, logits.contiguous(), train=need, saved=saved)
        if need:
            ctx.layer, ctx.saved, ctx.router = layer, saved, W_r is not None
            ctx.save_for_backward(x, W_r if W_r is not None else x)
        return y

    @staticmethod
    def backward(ctx, dy):
        # The backward reads the weight operands of the current masters: they
        # must not change between a forward and its backward (no optimizer
        # step in between), as in every usual training schedule.
        x, W_r = ctx.saved_tensors
        layer = ctx.layer
        g = layer.backward(dy.contiguous(), x, saved=ctx.saved)
        ctx.saved = None
        dW_r = None
        if ctx.router:
            dW_r = torch.empty_like(W_r)
            layer.router_backward(g["dlogits"], x, W_r.contiguous(), g["dx"], dW_r)
        return (g["dx"], None if ctx.router else g["dlogits"], dW_r, g["dW_gu"], g["dW_dn"], g["dWs_gu"],
                g["dWs_dn"], None)


class MoE(torch.nn.Module):
    """MoE layer for T tokens per call: E experts (gate/up [2m, d] and down
    [d, m] each, bf16 masters), top-k routing, optional BF16 shared expert of
    intermediate m_shared; fmt "mxfp8" or "bf16" for the routed experts.
    router=True adds router weights W_r [E, d] (forward(x)); otherwise the
    logits are given (forward(x, logits)).  aux_alpha > 0 adds the
    load-balancing term: its value after a forward is `aux_loss()` (a device
    scalar) and its gradient is applied inside the backward with weight 1, so
    it is not added to the loss again.  ring_rows / gather_sms select the
    dispatch ring (MXFP8)."""

    def __init__(self, T, d, m, E, k, fmt="mxfp8", m_shared=0, device="cuda", ring_rows=0, gather_sms=0,
                 router=False, aux_alpha=0.0):
        super().__init__()
        bf = dict(dtype=torch.bfloat16, device=device)
        self.W_r = torch.nn.Parameter(torch.empty(E, d, **bf).normal_(0.0, d ** -0.5)) if router else None
        self.W_gu = torch.nn.Parameter(torch.empty(E, 2 * m, d, **bf).normal_(0.0, d ** -0.5))
        self.W_dn = torch.nn.Parameter(torch.empty(E, d, m, **bf).normal_(0.0, m ** -0.5))
        if m_shared:
            self.Ws_gu = torch.nn.Parameter(torch.empty(2 * m_shared, d, **bf).normal_(0.0, d ** -0.5))
            self.Ws_dn = torch.nn.Parameter(torch.empty(d, m_shared, **bf).normal_(0.0, m_shared ** -0.5))
        else:
            self.Ws_gu = self.Ws_dn = None
        with torch.no_grad():
            shared = (self.Ws_gu, self.Ws_dn) if m_shared else None
            self.layer = MoELayer(T, d, m, E, k, fmt, shared=shared, backward=True, device=device,
                                  stacked=(self.W_gu, self.W_dn), ring_rows=ring_rows, gather_sms=gather_sms,
                                  aux_alpha=aux_alpha)

    def forward(self, x, logits=None):
        if (logits is None) != (self.W_r is not None):
            raise ValueError("pass logits exactly when the module has no router")
        return MoEFunction.apply(x, logits, self.W_r, self.W_gu, self.W_dn, self.Ws_gu, self.Ws_dn, self.layer)

    def aux_loss(self):
        """The load-balancing loss of the last forward (0-d fp32 device tensor)."""
        return self.layer.view(1, "aux", "f32", (1,))[0]
