"""Helpers shared by the GPU parity tests: build a layer from a workload
description, run the oracle on the same inputs, map padded GPU rows to the
oracle's expert-sorted rows."""
import numpy as np
import torch

import moe_inputs as mi
from oracle import moe as om
from oracle import numerics as nx


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


TOL = {"bf16": 5e-3, "mxfp8": 3e-2}


class Case:
    """Inputs drawn on the CPU (small workloads), a GPU layer, and oracle views."""

    def __init__(self, cfg, backward=False, device="cuda", flags=0):
        from mixture_experts_layer_device_gb300.layer import MoELayer
        self.cfg = cfg
        self.logits = mi.logits(cfg)
        self.x = mi.tokens(cfg)
        self.gu, self.dn = mi.experts(cfg)
        self.shared = mi.shared(cfg)
        self.dy = mi.out_grad(cfg)
        self.layer = MoELayer(cfg["T"], cfg["d"], cfg["m"], cfg["E"], cfg["k"], cfg["fmt"],
                              lambda e: (self.gu[e].to(device), self.dn[e].to(device)),
                              shared=None if self.shared is None else tuple(w.to(device) for w in self.shared),
                              backward=backward, device=device, flags=flags)
        self.xg = self.x.to(device)
        self.lg = self.logits.to(device)
        self.dyg = self.dy.to(device)

    def oracle_experts(self):
        gu = mi.to_f64(self.gu)
        dn = mi.to_f64(self.dn)
        return [(gu[e], dn[e]) for e in range(self.cfg["E"])]

    def oracle_shared(self):
        return None if self.shared is None else tuple(mi.to_f64(w) for w in self.shared)

    def route_views(self, which):
        """(counts, offsets, poff, inv) the GPU schedule wrote (numpy)."""
        E, R = self.cfg["E"], self.cfg["T"] * self.cfg["k"]
        L = self.layer
        return tuple(L.view(which, n, "i32", (s,)).cpu().numpy()
                     for n, s in (("counts", E), ("offsets", E + 1), ("poff", E + 1), ("inv", R)))

    def buffer(self, which, name):
        """Raw bytes (numpy uint8) of a named buffer."""
        import mixture_experts_layer_device_gb300 as pkg
        off, nb = pkg.moe_buffer_info(self.layer.cfg, which, name)
        base = self.layer.saved if which == 0 else self.layer.ws
        return base[off:off + nb].cpu().numpy()

    def oracle_forward(self):
        return om.forward(mi.to_f64(self.x), self.logits.numpy(), self.oracle_experts(), self.cfg["k"],
                          self.cfg["fmt"], shared=self.oracle_shared())


def padded_rows(counts, offsets, poff):
    """GPU padded row of each oracle (unpadded) expert-sorted row."""
    counts = np.asarray(counts)
    offsets = np.asarray(offsets)
    poff = np.asarray(poff)
    R = int(offsets[-1])
    e_of = np.repeat(np.arange(counts.size), counts)
    return poff[e_of] + np.arange(R) - offsets[e_of]


def unpack_tiled_scales(sf, rows, K):
    """Canonical [rows, K/32] scale bytes from the tiled layout (index permutation only)."""
    sf = np.asarray(sf, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    b = np.arange(K // 32)[None, :]
    off = ((r // 128) * (K // 128) + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (b % 4)
    return sf[off]


# ---------------------------------------------------------------- full-size sampling
def _prep_worker(args):
    e, gu, dn, fmt, backward = args
    return e, om.prepare_expert(gu.astype(np.float64), dn.astype(np.float64), fmt, backward)


class ExpertSubset:
    """experts[e] for the oracle holding only some experts (weights + prepared operands)."""

    def __init__(self, E, table):
        self.E, self.t = E, table

    def __len__(self):
        return self.E

    def __getitem__(self, e):
        return self.t[e]


def _compact(op):
    """A prepared operand held in fp32 where that represents it exactly
    (dequantised MXFP8 or bf16 values), else kept in float64 (NVFP4 values are
    divided by a second-level scale that is not a power of two); the oracle
    computes in fp64 either way."""
    o32 = np.asarray(op, dtype=np.float32)
    return o32 if np.array_equal(o32.astype(np.float64), op) else np.asarray(op, dtype=np.float64)


def prepare_subset(cfg, gu_all, dn_all, experts, backward):
    """Oracle S0 for some experts of device-resident bf16 masters (spawned
    worker pool).  With prepared operands the oracle reads the masters only for
    their shapes, so zero-stride stand-ins of the right shape replace them and
    the operands are kept in fp32: many experts fit in host memory."""
    import multiprocessing as mp
    import os
    experts = [int(e) for e in experts]
    table = {}
    nproc = max(1, min(len(experts), os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(nproc) as pool:
        for i in range(0, len(experts), nproc):          # bounded batches of masters in flight
            batch = experts[i:i + nproc]
            jobs = [(e, gu_all[e].float().cpu().numpy(), dn_all[e].float().cpu().numpy(), cfg["fmt"], backward)
                    for e in batch]
            for e, ops in pool.map(_prep_worker, jobs):
                shape_gu, shape_dn = tuple(gu_all[e].shape), tuple(dn_all[e].shape)
                table[e] = (np.broadcast_to(np.float64(0.0), shape_gu), np.broadcast_to(np.float64(0.0), shape_dn),
                            {k: _compact(v) for k, v in ops.items()})
    return ExpertSubset(cfg["E"], table)


# ---------------------------------------------------------------- streamed oracle experts
def _bf16_bits(t):
    """Raw bf16 bits of a device tensor as a host uint16 array (half the bytes of fp32)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _stream_worker(args):
    e, gu_bits, dn_bits, fmt, forward, backward = args
    ops = om.prepare_expert(nx.bf16_from_bits(gu_bits), nx.bf16_from_bits(dn_bits), fmt,
                            backward=backward, forward=forward)
    return e, {k: _compact(v) for k, v in ops.items()}


class StreamedExperts:
    """experts[e] for the oracle at the full workload sizes, prepared (S0) by a
    pool of spawned workers a bounded number of experts ahead, in the order the
    oracle asks for them (increasing expert index).  Host memory holds the
    operands of the expert in use plus the pool's read-ahead, not of all
    experts.  Each pass (forward, then backward) is announced with ``expect``:
    the experts it will ask for, in order, and which operand pair it needs."""

    def __init__(self, cfg, gu_all, dn_all):
        import multiprocessing as mp
        import os
        self.cfg, self.E = cfg, cfg["E"]
        self.gu_all, self.dn_all = gu_all, dn_all
        self.nproc = max(1, os.cpu_count() or 1)
        self.pool = mp.get_context("spawn").Pool(self.nproc)
        self.pending, self.queue = {}, []
        self.shape_gu = tuple(gu_all.shape[1:])
        self.shape_dn = tuple(dn_all.shape[1:])

    def expect(self, experts, forward, backward):
        assert not self.pending, "the previous pass did not consume every expert"
        self.queue = [int(e) for e in sorted(experts)]
        self.parts = (forward, backward)
        self._fill()

    def _fill(self):
        while self.queue and len(self.pending) < self.nproc + 2:
            e = self.queue.pop(0)
            job = (e, _bf16_bits(self.gu_all[e]), _bf16_bits(self.dn_all[e]), self.cfg["fmt"], *self.parts)
            self.pending[e] = self.pool.apply_async(_stream_worker, (job,))

    def __len__(self):
        return self.E

    def __getitem__(self, e):
        r = self.pending.pop(int(e))        # KeyError: an expert outside the announced pass
        _, ops = r.get()
        self._fill()
        return (np.broadcast_to(np.float64(0.0), self.shape_gu), np.broadcast_to(np.float64(0.0), self.shape_dn),
                ops)

    def close(self):
        self.pool.terminate()
        self.pool.join()
