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

    x [T, d] bf16, logits [T, E] fp32 -> y [T, d] bf16.  Backward returns dx,
    dlogits (fp32, zero outside each token's chosen experts) and the gradients
    of the bf16 masters."""

    @staticmethod
    def forward(ctx, x, logits, W_gu, W_dn, Ws_gu, Ws_dn, layer):
        layer.prepare_from(W_gu, W_dn, Ws_gu, Ws_dn)
        need = any(ctx.needs_input_grad[:6])
        saved = layer.new_saved() if need else None
        y = layer.forward(x.contiguous(), logits.contiguous(), train=need, saved=saved)
        if need:
            ctx.layer, ctx.saved = layer, saved
            ctx.save_for_backward(x)
        return y

    @staticmethod
    def backward(ctx, dy):
        # The backward reads the weight operands of the current masters: they
        # must not change between a forward and its backward (no optimizer
        # step in between), as in every usual training schedule.
        (x,) = ctx.saved_tensors
        g = ctx.layer.backward(dy.contiguous(), x.contiguous(), saved=ctx.saved)
        ctx.saved = None
        return g["dx"], g["dlogits"], g["dW_gu"], g["dW_dn"], g["dWs_gu"], g["dWs_dn"], None


class MoE(torch.nn.Module):
    """MoE layer for T tokens per call: E experts (gate/up [2m, d] and down
    [d, m] each, bf16 masters), top-k routing on given fp32 logits, optional
    BF16 shared expert of intermediate m_shared; fmt "mxfp8" or "bf16" for the
    routed experts.  ring_rows / gather_sms select the dispatch ring (MXFP8)."""

    def __init__(self, T, d, m, E, k, fmt="mxfp8", m_shared=0, device="cuda", ring_rows=0, gather_sms=0):
        super().__init__()
        bf = dict(dtype=torch.bfloat16, device=device)
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
                                  stacked=(self.W_gu, self.W_dn), ring_rows=ring_rows, gather_sms=gather_sms)

    def forward(self, x, logits):
        return MoEFunction.apply(x, logits, self.W_gu, self.W_dn, self.Ws_gu, self.Ws_dn, self.layer)
