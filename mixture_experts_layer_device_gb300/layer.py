"""Device-memory plumbing around the C ABI: owns the workspace / saved buffers
and the prepared expert weights (torch tensors), and calls the library.

All arithmetic (weight quantisation and transposes included) runs in the
library's CUDA kernels; torch only allocates memory and provides the stream.
"""
import torch

from . import (DTYPES, MOE_FLAG_BACKWARD, check, config, moe_backward, moe_buffer_info,
               moe_forward, moe_get_status, moe_padded_rows, moe_prepare_weights,
               moe_router_backward, moe_router_forward, moe_saved_bytes, moe_transpose_bf16,
               moe_workspace_bytes, weights)

_DT = {"i32": torch.int32, "f32": torch.float32, "bf16": torch.bfloat16, "u8": torch.uint8}


def _u8(nbytes, device):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


class MoELayer:
    """One MoE layer's prepared weights and buffers on one GPU.

    ``ring_rows`` > 0 (MXFP8) runs the forward's dispatch and gate/up GEMM as
    one persistent launch through a ring of that many rows, ``gather_sms`` of
    whose SMs gather (0 = the library default).  ``flags`` adds moe_config
    flag bits (the test hooks MOE_FLAG_DEBUG_STARVE / MOE_FLAG_DEBUG_DUMP).

    ``expert(e)`` returns the bf16 masters (W_gu [2m, d], W_dn [d, m]) of
    expert e as device tensors; they are converted expert by expert into the
    layout the kernels read (MXFP8 codes + prepared scales, and for the backward
    the per-expert transposed copies), so the masters never need to be
    resident all at once.  Alternatively ``stacked=(W_gu [E, 2m, d], W_dn
    [E, d, m])`` converts all experts with one launch per operand.
    """

    def __init__(self, T, d, m, E, k, fmt, expert=None, shared=None, backward=False, device="cuda",
                 stacked=None, ring_rows=0, gather_sms=0, aux_alpha=0.0, flags=0):
        self.T, self.d, self.m, self.E, self.k = T, d, m, E, k
        self.fmt = fmt
        self.mx = fmt == "mxfp8"
        self.nv = fmt == "nvfp4"          # forward only
        self.ms = 0 if shared is None else shared[1].shape[1]
        self.backward_enabled = backward
        self.device = device
        self.cfg = config(T, d, m, E, k, self.ms, DTYPES[fmt],
                          (MOE_FLAG_BACKWARD if backward else 0) | flags, ring_rows, gather_sms, aux_alpha)
        self.Rp = moe_padded_rows(self.cfg)
        self.ws = _u8(moe_workspace_bytes(self.cfg), device)
        self.saved = _u8(moe_saved_bytes(self.cfg), device) if backward else None
        self._prepare(expert, shared, stacked)

    # ------------------------------------------------------------ weights
    def _prepare(self, expert, shared, stacked=None):
        d, m, E, dev = self.d, self.m, self.E, self.device
        t = {}
        if self.nv:
            t["gu"] = torch.empty((E * 2 * m, d // 2), dtype=torch.uint8, device=dev)
            t["gu_scale"] = torch.empty((E * 2 * m * d // 16,), dtype=torch.uint8, device=dev)
            t["dn"] = torch.empty((E * d, m // 2), dtype=torch.uint8, device=dev)
            t["dn_scale"] = torch.empty((E * d * m // 16,), dtype=torch.uint8, device=dev)
            t["gu_gscale"] = torch.empty((E,), dtype=torch.float32, device=dev)
            t["dn_gscale"] = torch.empty((E,), dtype=torch.float32, device=dev)
        elif self.mx:
            t["gu"] = torch.empty((E * 2 * m, d), dtype=torch.uint8, device=dev)
            t["gu_scale"] = torch.empty((E * 2 * m * d // 32,), dtype=torch.uint8, device=dev)
            t["dn"] = torch.empty((E * d, m), dtype=torch.uint8, device=dev)
            t["dn_scale"] = torch.empty((E * d * m // 32,), dtype=torch.uint8, device=dev)
            if self.backward_enabled:
                t["gu_t"] = torch.empty((E * d, 2 * m), dtype=torch.uint8, device=dev)
                t["gu_t_scale"] = torch.empty((E * d * 2 * m // 32,), dtype=torch.uint8, device=dev)
                t["dn_t"] = torch.empty((E * m, d), dtype=torch.uint8, device=dev)
                t["dn_t_scale"] = torch.empty((E * m * d // 32,), dtype=torch.uint8, device=dev)
        else:
            t["gu"] = torch.empty((E, 2 * m, d), dtype=torch.bfloat16, device=dev)
            t["dn"] = torch.empty((E, d, m), dtype=torch.bfloat16, device=dev)
            if self.backward_enabled:
                t["gu_t"] = torch.empty((E, d, 2 * m), dtype=torch.bfloat16, device=dev)
                t["dn_t"] = torch.empty((E, m, d), dtype=torch.bfloat16, device=dev)
        self.tensors = t
        gsz, dsz = 2 * m * d, d * m
        if stacked is not None:
            gu, dn = (w.contiguous() for w in stacked)
            assert gu.shape == (E, 2 * m, d) and dn.shape == (E, d, m)
            if self.mx or self.nv:
                self.prepare_stacked(gu, dn)
            else:
                t["gu"].copy_(gu)
                t["dn"].copy_(dn)
                if self.backward_enabled:
                    check(moe_transpose_bf16(gu, E, 2 * m, d, t["gu_t"]))
                    check(moe_transpose_bf16(dn, E, d, m, t["dn_t"]))
        for e in range(E if stacked is None else 0):
            gu, dn = expert(e)
            assert gu.is_cuda and gu.dtype == torch.bfloat16 and gu.shape == (2 * m, d)
            assert dn.is_cuda and dn.dtype == torch.bfloat16 and dn.shape == (d, m)
            gu, dn = gu.contiguous(), dn.contiguous()
            if self.mx or self.nv:
                self._s0_q(gu, dn, 1, e, None)      # one expert into its slices of the operands
            else:
                t["gu"][e].copy_(gu)
                t["dn"][e].copy_(dn)
                if self.backward_enabled:
                    check(moe_transpose_bf16(gu, 1, 2 * m, d, t["gu_t"][e]))
                    check(moe_transpose_bf16(dn, 1, d, m, t["dn_t"][e]))
        if shared is not None:
            s_gu, s_dn = (w.contiguous() for w in shared)
            t["s_gu"], t["s_dn"] = s_gu, s_dn
            if self.backward_enabled:
                ms = self.ms
                t["s_gu_t"] = torch.empty((d, 2 * ms), dtype=torch.bfloat16, device=self.device)
                t["s_dn_t"] = torch.empty((ms, d), dtype=torch.bfloat16, device=self.device)
                check(moe_transpose_bf16(s_gu, 1, 2 * ms, d, t["s_gu_t"]))
                check(moe_transpose_bf16(s_dn, 1, d, ms, t["s_dn_t"]))
        self.tensors = t
        self.W = weights(**t)

    def prepare_stacked(self, gu, dn, stream=None):
        """S0 for all experts from stacked bf16 masters (W_gu [E, 2m, d],
        W_dn [E, d, m]) into this layer's MXFP8 or NVFP4 operands: one read of
        each master, which for an MXFP8 training layer also writes the
        backward's transposed copies.  Re-run after every update of the
        masters."""
        self._s0_q(gu, dn, self.E, 0, stream)

    def _s0_q(self, gu, dn, n, e0, stream):
        """S0 of n experts' masters (gu [n, 2m, d], dn [n, d, m]) straight into
        the operands of experts e0 .. e0 + n - 1 (codes, prepared scales and,
        with NVFP4, the second-level scales): one moe_prepare_weights call."""
        d, m, t, c = self.d, self.m, self.tensors, self.cfg
        cfg = c if n == self.E else config(c.T, d, m, n, 1, c.m_shared, c.dtype, 0)
        eb = 0.5 if self.nv else 1                      # code bytes per element
        sb = 16 if self.nv else 32                      # elements per scale byte
        og, od = e0 * 2 * m * d, e0 * d * m             # element offsets of the expert's matrices
        bw = self.backward_enabled and self.mx
        check(moe_prepare_weights(cfg, gu, dn, t["gu"].view(-1)[int(og * eb):], t["gu_scale"][og // sb:],
                                  t["dn"].view(-1)[int(od * eb):], t["dn_scale"][od // sb:],
                                  t["gu_t"].view(-1)[og:] if bw else None,
                                  t["gu_t_scale"][og // 32:] if bw else None,
                                  t["dn_t"].view(-1)[od:] if bw else None,
                                  t["dn_t_scale"][od // 32:] if bw else None,
                                  t["gu_gscale"][e0:] if self.nv else None,
                                  t["dn_gscale"][e0:] if self.nv else None, stream))

    def prepare_from(self, gu, dn, s_gu=None, s_dn=None, stream=None):
        """Re-derive every operand the kernels read from the current bf16
        masters (W_gu [E, 2m, d], W_dn [E, d, m], shared W_s_gu [2m_s, d],
        W_s_dn [d, m_s]): MXFP8 codes (both orientations for training) or bf16
        copies and transposes.  Run after every update of the masters."""
        E, d, m, t = self.E, self.d, self.m, self.tensors
        gu, dn = gu.contiguous(), dn.contiguous()
        if self.mx or self.nv:
            self.prepare_stacked(gu, dn, stream)
        else:
            t["gu"].copy_(gu)
            t["dn"].copy_(dn)
            if self.backward_enabled:
                check(moe_transpose_bf16(gu, E, 2 * m, d, t["gu_t"], stream))
                check(moe_transpose_bf16(dn, E, d, m, t["dn_t"], stream))
        if self.ms:
            t["s_gu"], t["s_dn"] = s_gu.contiguous(), s_dn.contiguous()
            if self.backward_enabled:
                check(moe_transpose_bf16(t["s_gu"], 1, 2 * self.ms, d, t["s_gu_t"], stream))
                check(moe_transpose_bf16(t["s_dn"], 1, d, self.ms, t["s_dn_t"], stream))
        self.W = weights(**t)

    def router_logits(self, x, W_r, logits=None, stream=None):
        """logits [T, E] fp32 = x W_r^T (the router projection)."""
        if logits is None:
            logits = torch.empty((self.T, self.E), dtype=torch.float32, device=self.device)
        check(moe_router_forward(self.cfg, x, W_r, logits, self.ws, stream))
        return logits

    def router_backward(self, dlogits, x, W_r, dx, dW_r, stream=None):
        """dx += bf16(dlogits) W_r in place (one rounding); dW_r = bf16(dlogits)^T x."""
        check(moe_router_backward(self.cfg, dlogits, x, W_r, dx, dW_r, self.ws, stream))

    def new_saved(self):
        """A fresh buffer for the activations one training forward keeps."""
        return _u8(moe_saved_bytes(self.cfg), self.device)

    # ------------------------------------------------------------ passes
    def forward(self, x, logits, y=None, train=False, stream=None, saved=None):
        if y is None:
            y = torch.empty((self.T, self.d), dtype=torch.bfloat16, device=self.device)
        if train and saved is None:
            if self.saved is None:
                raise ValueError("layer was built without backward support")
            saved = self.saved
        check(moe_forward(self.cfg, x, logits, self.W, y, saved if train else None, self.ws, stream))
        return y

    def alloc_grads(self):
        d, m, E, ms, dev = self.d, self.m, self.E, self.ms, self.device
        g = dict(dx=torch.empty((self.T, d), dtype=torch.bfloat16, device=dev),
                 dlogits=torch.empty((self.T, E), dtype=torch.float32, device=dev),
                 dW_gu=torch.empty((E, 2 * m, d), dtype=torch.bfloat16, device=dev),
                 dW_dn=torch.empty((E, d, m), dtype=torch.bfloat16, device=dev),
                 dWs_gu=None, dWs_dn=None)
        if ms:
            g["dWs_gu"] = torch.empty((2 * ms, d), dtype=torch.bfloat16, device=dev)
            g["dWs_dn"] = torch.empty((d, ms), dtype=torch.bfloat16, device=dev)
        return g

    def backward(self, dy, x, grads=None, stream=None, saved=None):
        g = grads or self.alloc_grads()
        check(moe_backward(self.cfg, dy, x, self.W, self.saved if saved is None else saved, g["dx"], g["dlogits"],
                           g["dW_gu"], g["dW_dn"], g["dWs_gu"], g["dWs_dn"], self.ws, stream))
        return g

    def status(self, stream=None):
        return moe_get_status(self.ws, stream)

    # ------------------------------------------------------------ inspection
    def view(self, which, name, dtype, shape):
        """Tensor view of a named sub-buffer of `saved` (which=0) or the workspace (1)."""
        off, nb = moe_buffer_info(self.cfg, which, name)
        base = self.saved if which == 0 else self.ws
        t = base[off:off + nb].view(_DT[dtype])
        n = 1
        for s in shape:
            n *= s
        return t[:n].view(*shape)
