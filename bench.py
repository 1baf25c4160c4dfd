#!/usr/bin/env python
"""Throughput of the GB300 mixture-of-experts layer (one JSON line on stdout).

A step is one pass of the layer's hot path over one batch of synthetic input:
route + schedule, dispatch, expert GEMMs with SwiGLU and MXFP8 quantisation,
shared expert, combine, and (for a fwd+bwd pass) the whole backward.  Expert
weight preparation (MXFP8 quantisation of the bf16 masters and the backward
copies) happens once per weight update, so it is timed separately ("s0_ms").

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--pass fwd|fwdbwd]
  python bench.py --impl reference ...     # the CPU oracle on a bounded sample

Default workload: the Kimi-K2.7-shaped layer (E=384, d=7168, m=2048, top-8,
T=16384, MXFP8 experts + BF16 shared expert of intermediate 2048), forward +
backward -- the one workload that runs every step of the path.  The layer
runs on one GPU and has no exchange step, so --gpus must be 1.
"""
import argparse
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s fwd & fwd+bwd on 1 GB300; % of GEMM/HBM roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
MX_OVER_BF16 = 2.0   # nominal dense MXFP8 : BF16 tensor-core ratio (4.5 : 2.25 PFLOP/s)
NV_OVER_MX = 3.0     # nominal dense NVFP4 : MXFP8 ratio (13.5 : 4.5 PFLOP/s)
# GB300's published dense peaks (context column of every fraction)
NOMINAL = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0, "mx_tflops": 4500.0, "nv_tflops": 13500.0}

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from an
# ncu capture, keyed by (workload, kernel).  An entry is removed whenever the
# kernel changes after the capture.
NCU_TRAFFIC = {
    # full-size launches of the timed step, one-pass capture of dram__bytes_read.sum and
    # dram__bytes_write.sum; the gate/up wgrad is the empty experts' zero fill plus the GEMM
    ("kimi-k2.7", "wgrad_gate_up"): (129_536 + 8_860_143_616) + (4_777_004_032 + 13_564_823_552),
    ("kimi-k2.7", "wgrad_down"): (103_168 + 4_397_457_920) + (1_658_128_640 + 6_752_918_272),
    ("kimi-k2.7", "gemm1_gate_up_swiglu"): 8_806_697_984 + 1_949_560_832,
    ("kimi-k2.7", "dgrad_gate_up"): 7_719_481_088 + 2_210_394_624,
    ("kimi-k2.7", "gemm2_down"): 3_839_812_864 + 2_203_856_128,
    ("deepseek-v4-pro", "gemm1_gate_up_swiglu"): 23_659_604_736 + 707_164_672,
    ("deepseek-v4-pro", "gemm2_down"): 9_965_006_592 + 2_929_535_232,
}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def workload(name):
    import moe_inputs as mi
    cfg = dict(mi.WORKLOADS[name])
    cfg["name"] = name
    return cfg


def active_experts(cfg):
    """Experts that receive rows (the step's routing, set by the bench after its
    warm-up; all E before): only their weights are read.  Every expert's dW is
    written, zeros for the empty ones."""
    return cfg.get("E_active", cfg["E"])


def experts_with_rows(layer, which):
    """Experts the layer's last routing gave rows to (its per-expert counts in
    `saved`, which=0, after a training forward, else in the workspace)."""
    counts = layer.view(which, "counts", "i32", (layer.E,))
    return int((counts > 0).sum().item())


def layer_work(cfg, passes):
    """Algorithmic FLOPs (split by arithmetic) and bytes of one step."""
    T, d, m, E, k, ms = (cfg[n] for n in ("T", "d", "m", "E", "k", "m_shared"))
    R = T * k
    mx = cfg["fmt"] == "mxfp8"
    mult = 3 if passes == "fwdbwd" else 1
    fl_exp = 6.0 * d * m * R * mult
    fl_sh = 6.0 * d * ms * T * mult
    wb = elem_bytes(cfg)                             # stored bytes per weight element
    wts = active_experts(cfg) * 3 * d * m * wb
    byt = wts + T * d * 2 + T * E * 4 + T * d * 2 + (3 * d * ms * 2 if ms else 0)
    if passes == "fwdbwd":
        byt += wts if mx else 0                      # backward operand copies
        byt += T * d * 2 * 2 + T * E * 4             # dy, dx, dlogits
        byt += E * 3 * d * m * 2 + 3 * d * ms * 2    # weight gradients (bf16)
        byt += 3 * d * ms * 2                        # shared weights re-read
    return fl_exp, fl_sh, byt


def elem_bytes(cfg):
    """Stored bytes per expert-operand element: MXFP8 1 + 1/32 (E8M0 per 32),
    NVFP4 1/2 + 1/16 (E4M3 per 16), BF16 2."""
    return {"mxfp8": 1 + 1 / 32, "nvfp4": 0.5 + 1 / 16}.get(cfg["fmt"], 2)


def kernel_work(cfg, name, train=False):
    """(FLOPs, algorithmic bytes, is_mx) of one step's launches of a traced
    kernel name (one launch per step for every GEMM and for the dispatch,
    combine and reverse kernels; the transposes and the route/schedule are
    several launches under one name).

    Bytes count every input read once and every output written once (x and
    dy once per token, not once per routed copy).  With MXFP8 experts a
    training pass's dispatch also writes the column-blocked codes of x, and its
    reverse combine both the row- and column-blocked codes of dO; the forward
    gate/up GEMM of a training pass saves G|U in bf16 and, with MXFP8, h as
    row- and column-blocked codes (with BF16, h in bf16)."""
    T, d, m, E, k, ms = (cfg[n] for n in ("T", "d", "m", "E", "k", "m_shared"))
    Ea = active_experts(cfg)               # weights read: experts with rows only
    R = T * k
    mx = cfg["fmt"] in ("mxfp8", "nvfp4")  # block-scaled expert operands
    a = elem_bytes(cfg)                    # bytes per stored expert operand element
    h_out = (R * 2 * m * 2 + (2 * R * m * a if mx else R * m * 2)) if train else R * m * a
    sh_out = (T * 2 * ms * 2 + T * ms * 2) if train else T * ms * 2
    tbl = {
        "gemm1_gate_up_swiglu": (2.0 * R * 2 * m * d, R * d * a + Ea * 2 * m * d * a + h_out, mx),
        "gemm2_down": (2.0 * R * d * m, R * m * a + Ea * d * m * a + R * d * 2, mx),
        "dgrad_down_swiglu_bwd": (2.0 * R * m * d, R * d * a + Ea * m * d * a + R * 2 * m * 2 * 2
                                  + (R * 2 * m * a if mx else 0), mx),
        "dgrad_gate_up": (2.0 * R * d * 2 * m, R * 2 * m * a + Ea * d * 2 * m * a + R * d * 2, mx),
        "wgrad_down": (2.0 * R * d * m, R * d * a + R * m * a + E * d * m * 2, mx),
        "wgrad_gate_up": (2.0 * R * 2 * m * d, R * 2 * m * a + R * d * a + E * 2 * m * d * 2, mx),
        "shared_gemm1_gate_up_swiglu": (2.0 * T * 2 * ms * d, T * d * 2 + 2 * ms * d * 2 + sh_out, False),
        "shared_gemm2_down": (2.0 * T * d * ms, T * ms * 2 + d * ms * 2 + T * d * 2, False),
        "shared_dgrad_down_swiglu_bwd": (2.0 * T * ms * d, T * d * 2 + ms * d * 2 + 2 * T * 2 * ms * 2, False),
        "shared_dgrad_gate_up": (2.0 * T * d * 2 * ms, T * 2 * ms * 2 + d * 2 * ms * 2 + T * d * 2, False),
        "shared_wgrad_down": (2.0 * T * d * ms, T * d * 2 + T * ms * 2 + d * ms * 2, False),
        "shared_wgrad_gate_up": (2.0 * T * 2 * ms * d, T * 2 * ms * 2 + T * d * 2 + 2 * ms * d * 2, False),
        "dispatch_gather": (0.0, T * d * 2 + R * d * a * (2 if mx and train else 1), mx),
        # ring: dispatch + gate/up GEMM in one launch; the ring itself stays on chip (L2)
        "quantize_tokens": (0.0, T * d * 2 + T * d * a, mx),
        "dispatch_xT": (0.0, T * d * 2 + R * d * a, mx),
        "dispatch_gemm1_ring": (2.0 * R * 2 * m * d, T * d * a + Ea * 2 * m * d * a + h_out, mx),
        "combine": (0.0, R * d * 2 + R * 8 + T * d * 2 * (2 if ms else 1), mx),
        "reverse_combine": (0.0, T * d * 2 + R * d * 2 + R * 8 + (2 * R * d * a if mx else R * d * 2), mx),
        "reverse_dispatch": (0.0, R * d * 2 + R * 8 + T * d * 2 * (2 if ms else 1) + T * E * 4, mx),
        "route_schedule": (0.0, T * E * 4 + R * 4 * 6, mx),
        # MXFP8: dGU^T only (x^T, dO^T and h^T come from the dispatch, B1 and S4)
        "transpose_wgrad_operands": (0.0, (R * 2 * m * (2 + a)) if mx
                                     else (R * 2 * m + R * m + 2 * R * d) * (2 + a), mx),
        "shared_transpose_wgrad_operands": (0.0, 2 * 2 * T * (ms + d + 2 * ms + d), False),
    }
    return tbl.get(name)


def output_bytes(cfg, name):
    """Bytes a kernel name writes per step when its output write dominates (the
    expert weight gradients write bf16 dW for every expert)."""
    d, m, E = cfg["d"], cfg["m"], cfg["E"]
    return {"wgrad_gate_up": E * 2 * m * d * 2, "wgrad_down": E * d * m * 2}.get(name)


def kernels_in_region(name, cfg, train):
    """Kernel launches inside one traced region of the library: route + the
    three schedule kernels; with MXFP8 experts the dispatch and the reverse
    combine also run the one-block tile-order sort first, and an inference
    dispatch quantises every token once before it; the balance term is a
    partial and a finishing kernel."""
    mx = cfg["fmt"] == "mxfp8"
    if name == "route_schedule":
        return 4
    if name == "dispatch_gather" and mx:
        return 2 if train else 3
    if name in ("reverse_combine", "dispatch_xT") and mx:
        return 2
    if name in ("wgrad_gate_up", "wgrad_down") and mx:   # + the empty experts' zero fill
        return 2
    if name == "balance_loss":
        return 2
    return 1


def write_probe_gbs(dev):
    """Write-only HBM bandwidth of this GPU: a device fill of 8 GB (taken
    before the timed region; context for write-dominated kernels).  The fill
    runs on 8-byte elements: torch's fill of 1- and 2-byte elements issues
    narrow stores and reaches only about half the write bandwidth."""
    import torch
    buf = torch.empty(1 << 30, dtype=torch.int64, device=dev)
    buf.zero_()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(3):
        buf.zero_()
    b.record()
    b.synchronize()
    gbs = 3 * buf.numel() * 8 / (a.elapsed_time(b) / 1e3) / 1e9
    del buf
    torch.cuda.empty_cache()
    return gbs


def mxfp8_peak_probe(dev):
    """Dense MXFP8 GEMM rate of this GPU: the vendor library's block-scaled
    E4M3 GEMM (torch._scaled_mm with E8M0 scales) at 8192^3, as a burst (best
    of 10 single calls) and sustained (calls back to back for about 3 s, under
    the power cap).  Taken before the timed region; None fields if the library
    path is unavailable."""
    import torch
    M = N = K = 8192
    try:
        g = torch.Generator(device=dev).manual_seed(0)
        a = torch.randn((M, K), device=dev, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn((N, K), device=dev, generator=g).to(torch.float8_e4m3fn)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        best, f_best = float("inf"), None
        for shape_a, shape_b in (((M * K // 32,), (N * K // 32,)), ((M, K // 32), (N, K // 32))):
            sa = torch.full(shape_a, 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
            sb = torch.full(shape_b, 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)

            def f(sa=sa, sb=sb):
                return torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)

            try:
                for _ in range(3):
                    f()
                torch.cuda.synchronize()
            except Exception:     # this scale layout is not accepted by this torch build
                continue
            for _ in range(10):
                ev[0].record()
                f()
                ev[1].record()
                ev[1].synchronize()
                ms = ev[0].elapsed_time(ev[1])
                if ms < best:
                    best, f_best = ms, f
        if f_best is None:
            raise RuntimeError("no block-scaled MXFP8 GEMM path")
        f = f_best
        n, t0 = 0, time.time()
        ev[0].record()
        while time.time() - t0 < 3.0:
            for _ in range(20):
                f()
            n += 20
            torch.cuda.synchronize()
        ev[1].record()
        ev[1].synchronize()
        sus = ev[0].elapsed_time(ev[1]) / n
        fl = 2.0 * M * N * K
        return {"burst_tflops": round(fl / (best / 1e3) / 1e12, 1), "sustained_tflops": round(fl / (sus / 1e3) / 1e12, 1),
                "how": "torch._scaled_mm E4M3 x E4M3 with E8M0 block scales (vendor library), 8192^3, flat and 2-D "
                       "scale tensors; burst = best of 10 calls each, sustained = back to back for 3 s"}
    except Exception as exc:  # no block-scaled library path here: fall back, and say so
        return {"burst_tflops": None, "sustained_tflops": None, "how": "unavailable: %s" % str(exc)[:160]}


def tensor_peaks(peaks, peaks_src, mxp):
    """Denominators of every fraction: HBM copy bandwidth, BF16 and MXFP8
    dense tensor rates, each measured on this GPU.  The primary fraction uses
    the burst rates (the stricter ones); sustained and published-nominal
    fractions are reported beside it."""
    P = {"hbm": peaks["hbm_gbs"], "bf16": peaks["bf16_tflops"], "bf16_s": peaks["bf16_tflops_sustained"],
         "src": peaks_src}
    if mxp and mxp.get("burst_tflops"):
        P.update(mx=mxp["burst_tflops"], mx_s=mxp["sustained_tflops"], mx_src="measured MXFP8 GEMM (%s)" % mxp["how"])
    else:
        P.update(mx=MX_OVER_BF16 * P["bf16"], mx_s=MX_OVER_BF16 * P["bf16_s"],
                 mx_src="%.0f x %s BF16 (MXFP8 probe unavailable)" % (MX_OVER_BF16, peaks_src))
    # no NVFP4 GEMM rate is measured here: the nominal dense ratio to MXFP8
    P.update(nv=NV_OVER_MX * P["mx"], nv_s=NV_OVER_MX * P["mx_s"],
             nv_src="%.0f x the MXFP8 rate above (nominal dense NVFP4 : MXFP8, 13.5 : 4.5; no NVFP4 GEMM measured)"
                    % NV_OVER_MX)
    return P


def _tensor_peak(cfg, mx, P, kind=""):
    """(peak, sustained peak, nominal peak) of a kernel's arithmetic."""
    if not mx:
        return P["bf16"], P["bf16_s"], NOMINAL["bf16_tflops"]
    if cfg["fmt"] == "nvfp4":
        return P["nv"], P["nv_s"], NOMINAL["nv_tflops"]
    return P["mx"], P["mx_s"], NOMINAL["mx_tflops"]


def kernel_roofline(cfg, name, train, ms_per_step, P):
    """Bound, achieved and peak of one kernel: the larger of its tensor time
    (FLOPs at the tensor peak of its arithmetic) and its HBM time (algorithmic
    bytes at the copy bandwidth) names the bound.  `frac_sustained` and
    `frac_nominal` divide the same achieved rate by the sustained tensor rate
    and by GB300's published dense peaks."""
    w = kernel_work(cfg, name, train)
    if w is None or ms_per_step <= 0:
        return None
    flops, byts, mx = w
    tpeak, tpeak_s, tpeak_n = _tensor_peak(cfg, mx, P)
    t_tensor = flops / (tpeak * 1e12)
    t_hbm = byts / (P["hbm"] * 1e9)
    sec = ms_per_step / 1e3
    if t_tensor >= t_hbm:
        ach = flops / sec / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": tpeak, "unit": "TFLOP/s", "mx": mx,
                "frac": ach / tpeak, "frac_sustained": ach / tpeak_s, "frac_nominal": ach / tpeak_n,
                "t_tensor_ms": t_tensor * 1e3, "t_hbm_ms": t_hbm * 1e3}
    ach = byts / sec / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": P["hbm"], "unit": "GB/s", "mx": mx,
            "frac": ach / P["hbm"], "frac_sustained": ach / P["hbm"], "frac_nominal": ach / NOMINAL["hbm_gbs"],
            "t_tensor_ms": t_tensor * 1e3, "t_hbm_ms": t_hbm * 1e3}


def layer_roofline(cfg, passes, ms_step, P):
    """The whole step against max(FLOPs / tensor peak, algorithmic bytes / HBM):
    `frac` at the measured burst rates, beside it at the sustained rates and at
    GB300's published dense peaks."""
    fl_exp, fl_sh, byt = layer_work(cfg, passes)
    pk, pk_s, pk_n = _tensor_peak(cfg, cfg["fmt"] != "bf16", P)

    def roof(t_exp, t_bf, hbm):
        t_t = fl_exp / t_exp / 1e12 + fl_sh / t_bf / 1e12
        t_h = byt / hbm / 1e9
        return max(t_t, t_h), t_t, t_h

    t_roof, t_tensor, t_hbm = roof(pk, P["bf16"], P["hbm"])
    t_s = roof(pk_s, P["bf16_s"], P["hbm"])[0]
    t_n = roof(pk_n, NOMINAL["bf16_tflops"], NOMINAL["hbm_gbs"])[0]
    sec = ms_step / 1e3
    return {"tokens_per_s": round(cfg["T"] / t_roof, 1), "frac": round(t_roof / sec, 4),
            "experts_with_rows": active_experts(cfg),
            "frac_sustained": round(t_s / sec, 4), "frac_nominal": round(t_n / sec, 4),
            "bound": "tensor" if t_tensor >= t_hbm else "hbm", "t_tensor_ms": round(t_tensor * 1e3, 3),
            "t_hbm_ms": round(t_hbm * 1e3, 3),
            "peaks": "HBM %.1f GB/s, BF16 %.1f TFLOP/s (%s, burst), %s"
                     % (P["hbm"], P["bf16"], P["src"],
                        ("NVFP4 %.1f TFLOP/s (%s)" % (P["nv"], P["nv_src"])) if cfg["fmt"] == "nvfp4"
                        else "MXFP8 %.1f TFLOP/s (%s)" % (P["mx"], P["mx_src"]))}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        # the first sample is on file before the caller starts timing (at most 3 s)
        t0 = time.time()
        while self.p is not None and self.p.poll() is None and time.time() - t0 < 3.0:
            if os.path.getsize(self.f.name) > 0:
                break
            time.sleep(0.05)

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        self.f.close()
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


REJECTING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clk):
    """Whether a timed region's clock record disqualifies its number: a
    hardware or thermal slowdown was active, or the SM clock sat well below its
    maximum with no reason given (a clock lock left by someone else).
    sw_power_cap alone is normal under a dense load and is kept."""
    if any(r in clk.get("reasons", []) for r in REJECTING_REASONS):
        return True
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    return bool(sm and smax and sm < 0.8 * smax and not clk.get("reasons"))


def gpu_index():
    """nvidia-smi index of the device torch calls cuda:0."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if ids and ids[0].isdigit():
            return int(ids[0])
    return 0


# ----------------------------------------------------------------------------- oracle (CPU)
def _prep_worker(args):
    import numpy as np
    from oracle import moe as om
    e, gu, dn, fmt, forward, backward = args
    ops = om.prepare_expert(gu.astype(np.float64), dn.astype(np.float64), fmt, backward=backward, forward=forward)
    out = {}
    for key, v in ops.items():                  # held in fp32 where that is exact (the oracle computes in fp64)
        v32 = v.astype(np.float32)
        out[key] = v32 if np.array_equal(v32, v) else v
    return e, out


class _Experts:
    """experts[e] view for the oracle: only the sample's experts are held."""

    def __init__(self, E, table):
        self.E, self.t = E, table

    def __len__(self):
        return self.E

    def __getitem__(self, e):
        return self.t[e]


def oracle_sample(cfg, passes, x_dev, logits_dev, dy_dev, n_tok):
    """Host copies of an n_tok-token seeded sample and of its experts' masters."""
    import moe_inputs as mi
    from oracle import moe as om
    tok = mi.sample_tokens(cfg, n_tok)
    lg = logits_dev[tok].cpu().numpy()
    idx, _ = om.route(lg, cfg["k"])
    need = sorted(set(int(e) for e in idx.reshape(-1)))
    masters = {}
    for e in need:
        gu, dn = mi.expert(cfg, e, device=x_dev.device)
        masters[e] = (gu.float().cpu().numpy(), dn.float().cpu().numpy())
    sh = mi.shared(cfg, device=x_dev.device)
    shared = None if sh is None else tuple(mi.to_f64(w) for w in sh)
    return dict(tok=tok, x=mi.to_f64(x_dev[tok]), logits=lg, dy=None if dy_dev is None else mi.to_f64(dy_dev[tok]),
                need=need, masters=masters, shared=shared, passes=passes)


def oracle_dw_sample(cfg, layer, x_dev, dy_dev, n=4, max_rows=2048):
    """Host copies for the oracle's weight gradients of n seeded experts over all
    their rows (experts with 1..max_rows rows, so the sample stays within
    seconds): each expert's tokens, combine weights and masters, from the
    layer's routing of the bench's own inputs."""
    import numpy as np
    import moe_inputs as mi
    T, k, E = cfg["T"], cfg["k"], cfg["E"]
    counts = layer.view(0, "counts", "i32", (E,)).cpu().numpy()
    idx = layer.view(0, "idx", "i32", (T, k)).cpu().numpy().reshape(-1)
    w = layer.view(0, "w", "f32", (T, k)).cpu().numpy().reshape(-1).astype(np.float64)
    rows, masters = {}, {}
    for e in mi.sample_experts(counts, cfg["seed"], n=n, max_rows=max_rows):
        e = int(e)
        slots = np.nonzero(idx == e)[0]
        toks = slots // k
        t_dev = __import__("torch").as_tensor(toks, device=x_dev.device)
        rows[e] = (mi.to_f64(x_dev[t_dev]), mi.to_f64(dy_dev[t_dev]), w[slots])
        gu, dn = mi.expert(cfg, e, device=x_dev.device)
        masters[e] = (gu.float().cpu().numpy(), dn.float().cpu().numpy())
    return dict(rows=rows, masters=masters, passes="fwdbwd", need=sorted(rows))


def oracle_prepare(cfg, sample):
    """Weight preparation (S0) of the sample's experts by the oracle, in parallel
    (the masters themselves are not kept: with prepared operands the oracle
    reads them only for their shapes)."""
    import numpy as np
    bwd = sample["passes"] == "fwdbwd"
    jobs = [(e, gu, dn, cfg["fmt"], True, bwd) for e, (gu, dn) in sample["masters"].items()]
    t0 = time.perf_counter()
    nproc = max(1, min(len(jobs), os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(nproc) as pool:
        ops = dict(pool.map(_prep_worker, jobs))
    table = {e: (np.broadcast_to(np.float64(0.0), sample["masters"][e][0].shape),
                 np.broadcast_to(np.float64(0.0), sample["masters"][e][1].shape), ops[e]) for e in ops}
    sample["masters"] = None
    return _Experts(cfg["E"], table), time.perf_counter() - t0


def blas_threads(n):
    """Sets the thread count of numpy's OpenBLAS in this process through the
    library's own setter (ctypes); returns the previous count, or None where no
    such library or setter is found."""
    import ctypes
    import glob
    import numpy
    root = os.path.dirname(numpy.__file__)
    libs = glob.glob(os.path.join(os.path.dirname(root), "numpy.libs", "*openblas*")) + \
        glob.glob(os.path.join(root, ".libs", "*openblas*"))
    for path in libs:
        try:
            L = ctypes.CDLL(path)
        except OSError:
            continue
        for sfx in ("scipy_openblas_%s_num_threads64_", "openblas_%s_num_threads64_", "openblas_%s_num_threads"):
            if hasattr(L, sfx % "set") and hasattr(L, sfx % "get"):
                prev = getattr(L, sfx % "get")()
                getattr(L, sfx % "set")(int(n))
                return prev
    return None


def oracle_step(cfg, passes, sample, experts):
    from oracle import moe as om
    y, saved = om.forward(sample["x"], sample["logits"], experts, cfg["k"], cfg["fmt"], shared=sample["shared"])
    if passes == "fwdbwd":
        om.backward(sample["dy"], sample["x"], experts, cfg["k"], cfg["fmt"], saved, shared=sample["shared"],
                    dw_experts=sample["need"])
    return y


def oracle_sample_desc(cfg, passes, n_tok, n_exp):
    return ("%d seeded token(s) of the %s workload (%s): route, the %d experts they select, %scombine%s, "
            "float64 NumPy; expert weight preparation (MXFP8 quantisation, S0) done beforehand like the "
            "GPU side"
            % (n_tok, cfg["name"], "fwd+bwd" if passes == "fwdbwd" else "fwd", n_exp,
               "shared expert, " if cfg["m_shared"] else "",
               ", full backward incl. the sample's weight gradients" if passes == "fwdbwd" else ""))


# ----------------------------------------------------------------------------- main arms
def build_inputs(cfg, device, passes):
    import torch
    import moe_inputs as mi
    x = mi.tokens(cfg, device)
    logits = mi.logits(cfg, device)
    dy = mi.out_grad(cfg, device) if passes == "fwdbwd" else None
    E, d, m = cfg["E"], cfg["d"], cfg["m"]
    gu_all = torch.empty((E, 2 * m, d), dtype=torch.bfloat16, device=device)
    dn_all = torch.empty((E, d, m), dtype=torch.bfloat16, device=device)
    for e in range(E):
        gu_all[e], dn_all[e] = mi.expert(cfg, e, device)
    shared = mi.shared(cfg, device)
    return x, logits, dy, gu_all, dn_all, shared


def time_s0(layer, gu_all, dn_all, stream):
    """Weight preparation of all experts (the same kernels the layer was built with)."""
    import torch
    import mixture_experts_layer_device_gb300 as pkg
    E, d, m = layer.E, layer.d, layer.m
    t = layer.tensors

    def run():
        if layer.mx or layer.nv:
            layer.prepare_stacked(gu_all, dn_all, stream=stream)
        elif layer.backward_enabled:
            pkg.check(pkg.moe_transpose_bf16(gu_all, E, 2 * m, d, t["gu_t"], stream))
            pkg.check(pkg.moe_transpose_bf16(dn_all, E, d, m, t["dn_t"], stream))

    run()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b)


def workload_desc(cfg, bwd, layer=None):
    mx = cfg["fmt"] == "mxfp8"
    ring = layer.cfg.ring_rows if layer is not None else 0
    return {"workload": cfg["name"], "pass": "fwd+bwd" if bwd else "fwd", "T": cfg["T"], "d": cfg["d"],
            "m": cfg["m"], "E": cfg["E"], "k": cfg["k"], "m_shared": cfg["m_shared"],
            "experts": cfg["fmt"], "router_bias": cfg["bias"], "parallelism": "1gpu",
            "dispatch": ("ring of %d rows, %d gather SMs" % (ring, layer.cfg.gather_sms or 8)
                         if ring else "materialised"),
            "l2": "inputs larger than L2 (%.1f GB of expert weights stored)"
                  % (3 * cfg["E"] * cfg["d"] * cfg["m"] * elem_bytes(cfg) / 1e9)}


def summarize(cfg, train, recs, steps, total_ms, P, write_gbs):
    """Per-kernel breakdown of a traced timed region (the library's event trace:
    (name, ms) per traced launch), the dominant kernel's roofline and the
    number of kernel launches."""
    per = {}
    launches = 0
    for name, ms in recs:
        c, t = per.get(name, (0, 0.0))
        per[name] = (c + 1, t + ms)
        launches += kernels_in_region(name, cfg, train)
    kernel_total = sum(t for _, t in per.values()) or 1.0
    dom = max(per.items(), key=lambda kv: kv[1][1])[0]
    cnt, tot = per[dom]
    kr = kernel_roofline(cfg, dom, train, tot / steps, P)
    if kr is None:
        roof = {"kernel": dom, "bound": None, "achieved": None, "peak": None, "unit": None, "frac": None,
                "traffic": None}
    else:
        if kr["bound"] == "tensor":
            note = ((P["nv_src"] if cfg["fmt"] == "nvfp4" else P["mx_src"]) if kr["mx"]
                    else "%s BF16 GEMM, burst" % P["src"])
        else:
            note = "%s HBM copy bandwidth" % P["src"]
        ob = output_bytes(cfg, dom)
        roof = {"kernel": dom, "bound": kr["bound"], "achieved": round(kr["achieved"], 1), "peak": round(kr["peak"], 1),
                "unit": kr["unit"], "frac": round(kr["frac"], 4), "frac_sustained": round(kr["frac_sustained"], 4),
                "frac_nominal": round(kr["frac_nominal"], 4), "traffic": NCU_TRAFFIC.get((cfg["name"], dom)),
                "peak_source": note, "launch_ms": round(tot / cnt, 4),
                "write_probe": None if ob is None else {
                    "note": "output-write-dominated kernel: its bf16 dW write rate against this GPU's "
                            "write-only bandwidth (device fill of 8 GB, measured before the timed region)",
                    "written_gbs": round(ob / (tot / steps / 1e3) / 1e9, 1), "fill_gbs": round(write_gbs, 1),
                    "frac": round(ob / (tot / steps / 1e3) / 1e9 / write_gbs, 4)}}
    kernels = {}
    for n, (c, t) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        kernels[n] = {"launches_per_step": c / steps, "ms_per_step": round(t / steps, 4),
                      "share": round(t / kernel_total, 4)}
        r = kernel_roofline(cfg, n, train, t / steps, P)
        if r is not None:
            kernels[n].update({"bound": r["bound"], "frac": round(r["frac"], 4),
                               "frac_sustained": round(r["frac_sustained"], 4),
                               "frac_nominal": round(r["frac_nominal"], 4)})
    rs = per.get("route_schedule", (0, 0.0))[1] / kernel_total
    return {"roofline": roof, "kernels": kernels, "route_schedule_share": round(rs, 4),
            "gpu_launches": launches}


def timed_region(stream, fn, K, trace=False):
    """K calls of fn between CUDA events on `stream`, synchronised on both
    sides; with `trace`, the library's per-launch event records as well."""
    import torch
    import mixture_experts_layer_device_gb300 as pkg
    if trace:
        pkg.check(pkg.moe_trace_enable(K * 64 + 64))
        pkg.moe_trace_clear()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K):
        fn()
    b.record(stream)
    b.synchronize()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    recs = pkg.moe_trace_records() if trace else []
    if trace:
        pkg.moe_trace_enable(0)
    return ms, recs


TARGET = "deepseek-v4-pro"


def run_target(args, P):
    """The target leg: the MXFP8 forward of the largest workload (DeepSeek-V4-Pro
    shape, 8 hot experts), built after the main workload's buffers are freed,
    with its own timed region, clock record, per-kernel trace and rooflines."""
    import torch
    from mixture_experts_layer_device_gb300.layer import MoELayer
    cfg = workload(TARGET)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    x, logits, _, gu_all, dn_all, shared = build_inputs(cfg, dev, "fwd")
    layer = MoELayer(cfg["T"], cfg["d"], cfg["m"], cfg["E"], cfg["k"], cfg["fmt"], shared=shared, backward=False,
                     device=dev, stacked=(gu_all, dn_all))
    del gu_all, dn_all
    torch.cuda.empty_cache()
    y = torch.empty((cfg["T"], cfg["d"]), dtype=torch.bfloat16, device=dev)

    def step():
        layer.forward(x, logits, y=y, train=False, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if layer.status() != 0:
        raise RuntimeError("device status after the target leg's warm-up")
    cfg["E_active"] = experts_with_rows(layer, 1)
    clocks = Clocks(gpu_index())
    total_ms, _ = timed_region(stream, step, args.steps)
    clk = clocks.stop()
    if clocks_rejected(clk):
        first = clk
        clocks = Clocks(gpu_index())
        total_ms, _ = timed_region(stream, step, args.steps)
        clk = clocks.stop()
        clk["remeasured_after"] = {"sm_mhz": first["sm_mhz"], "reasons": first["reasons"]}
    _, recs = timed_region(stream, step, args.steps, trace=True)
    if layer.status() != 0:
        raise RuntimeError("device status after the target leg")
    ms = total_ms / args.steps
    summ = summarize(cfg, False, recs, args.steps, total_ms, P, 0.0)
    ring = ring_leg(args, cfg, P, layer, x, logits, y, stream)
    return {"note": "MXFP8 forward of the largest workload; target: layer_roofline.frac >= 0.60",
            "value": round(cfg["T"] / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "steps": args.steps, "warmup": args.warmup, "config": workload_desc(cfg, False, layer),
            "layer_roofline": layer_roofline(cfg, "fwd", ms, P), "roofline": summ["roofline"],
            "kernels": summ["kernels"], "route_schedule_share": summ["route_schedule_share"],
            "gpu_launches": summ["gpu_launches"], "clocks": clk, "ring": ring}


def ring_leg(args, cfg, P, layer, x, logits, y_ref, stream, ring_rows=8192, gather_sms=8):
    """The same forward through the persistent ring kernel: one cooperative
    launch in which gather SMs copy the expert-sorted rows into a ring of
    ring_rows rows that the other SMs' gate/up GEMM consumes, so the dispatched
    rows are never materialised.  Timed after the materialised leg, on the same
    weights and inputs; its output must equal that leg's bit for bit."""
    import torch
    import mixture_experts_layer_device_gb300 as pkg
    c = layer.cfg
    rc = pkg.MoeConfig(c.T, c.d, c.m, c.E, c.k, c.m_shared, c.dtype, c.flags, ring_rows, gather_sms)
    ws = torch.empty(pkg.moe_workspace_bytes(rc), dtype=torch.uint8, device=x.device)
    y = torch.empty_like(y_ref)

    def step():
        pkg.check(pkg.moe_forward(rc, x, logits, layer.W, y, None, ws, stream))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    total_ms, _ = timed_region(stream, step, args.steps)
    st = pkg.moe_get_status(ws)
    if st != 0:
        raise RuntimeError("device status %d after the ring leg" % st)
    ms = total_ms / args.steps
    return {"ms_per_step": round(ms, 4), "tokens_per_s": round(cfg["T"] / (ms / 1e3), 1),
            "ring_rows": ring_rows, "gather_sms": gather_sms,
            "workspace_gb": round(ws.numel() / 1e9, 3), "materialised_workspace_gb": round(layer.ws.numel() / 1e9, 3),
            "layer_roofline_frac": layer_roofline(cfg, "fwd", ms, P)["frac"],
            "bitwise_equal_to_materialised": bool(torch.equal(y.view(torch.int16), y_ref.view(torch.int16)))}


def run_ours(args, cfg, passes):
    import numpy as np
    import torch
    import mixture_experts_layer_device_gb300 as pkg
    from mixture_experts_layer_device_gb300.layer import MoELayer

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peaks_src = load_peaks()
    mxp = None if args.profile_run else mxfp8_peak_probe(dev)   # profiler launch lists stay the layer's
    P = tensor_peaks(peaks, peaks_src, mxp)

    x, logits, dy, gu_all, dn_all, shared = build_inputs(cfg, dev, passes)
    bwd = passes == "fwdbwd"
    ring_rows = args.ring if cfg["fmt"] == "mxfp8" else 0
    layer = MoELayer(cfg["T"], cfg["d"], cfg["m"], cfg["E"], cfg["k"], cfg["fmt"], shared=shared, backward=bwd,
                     device=dev, stacked=(gu_all, dn_all), ring_rows=ring_rows, gather_sms=args.gather_sms)
    s0_ms = time_s0(layer, gu_all, dn_all, stream)
    sample = None
    want_cpu = not args.no_cpu_baseline and not args.profile_run
    n_tok = 1 if bwd else 4
    sample256 = None
    if want_cpu:
        sample = oracle_sample(cfg, passes, x, logits, dy, n_tok)
        sample256 = oracle_sample(cfg, "fwd", x, logits, None, 256)
    keep_masters = bwd and layer.mx      # re-quantised every update in the with-S0 step
    if not keep_masters:
        del gu_all, dn_all
        torch.cuda.empty_cache()

    grads = layer.alloc_grads() if bwd else None
    y = torch.empty((cfg["T"], cfg["d"]), dtype=torch.bfloat16, device=dev)

    def step():
        layer.forward(x, logits, y=y, train=bwd, stream=stream)
        if bwd:
            layer.backward(dy, x, grads=grads, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = layer.status()
    if st != 0:
        raise RuntimeError("device status %d after warm-up" % st)
    cfg["E_active"] = experts_with_rows(layer, 0 if bwd else 1)
    dw_sample = oracle_dw_sample(cfg, layer, x, dy) if (want_cpu and bwd) else None

    def timed(fn, K, trace=False):
        return timed_region(stream, fn, K, trace)

    write_gbs = write_probe_gbs(dev)
    clocks = Clocks(gpu_index())
    if args.profile_run:      # a single, traced timed region (short profiler launch lists)
        total_ms, recs = timed(step, args.steps, trace=True)
        clk = clocks.stop()
    else:
        total_ms, _ = timed(step, args.steps)
        clk = clocks.stop()
        # measured once more if the clock record rejects it; the second record
        # is reported
        if clocks_rejected(clk):
            first = clk
            clocks = Clocks(gpu_index())
            total_ms, _ = timed(step, args.steps)
            clk = clocks.stop()
            clk["remeasured_after"] = {"sm_mhz": first["sm_mhz"], "reasons": first["reasons"]}
        # per-kernel breakdown from a second, traced run (its event records would
        # add gaps between launches to the headline timing)
        _, recs = timed(step, args.steps, trace=True)
    ms_step = total_ms / args.steps
    tokens = cfg["T"]
    value = tokens * args.steps / (total_ms / 1e3)

    fwd_value = value
    if args.profile_run:      # one timed region only (keeps profiler launch lists short)
        per_ms = {}
        for name, ms in recs:
            per_ms[name] = per_ms.get(name, 0.0) + ms
        return {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "ms_per_step": round(ms_step, 4),
                "config": {"workload": cfg["name"], "T": cfg["T"], "E": cfg["E"]}, "profile_run": True,
                "kernels_ms_per_step": {n: round(t / args.steps, 4) for n, t in per_ms.items()}}, P
    if bwd:
        fms, _ = timed(lambda: layer.forward(x, logits, y=y, train=False, stream=stream), args.steps)
        fwd_value = tokens * args.steps / (fms / 1e3)
    # the same step captured once into a CUDA graph and replayed (no host
    # launch overhead; context for small workloads)
    graph_info = None
    try:
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            layer.forward(x, logits, y=y, train=bwd, stream=side)
            if bwd:
                layer.backward(dy, x, grads=grads, stream=side)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cs = torch.cuda.current_stream()
            layer.forward(x, logits, y=y, train=bwd, stream=cs)
            if bwd:
                layer.backward(dy, x, grads=grads, stream=cs)
        graph.replay()
        torch.cuda.synchronize()
        g_ms, _ = timed(graph.replay, args.steps)
        graph_info = {"ms_per_step": round(g_ms / args.steps, 4),
                      "tokens_per_s": round(tokens * args.steps / (g_ms / 1e3), 1)}
        del graph
    except Exception as exc:  # capture unsupported here: report, do not fail the run
        graph_info = {"unavailable": str(exc)[:200]}
    with_s0 = None
    if keep_masters:
        # a training update re-quantises the bf16 masters (S0, both orientations)
        # before its forward+backward
        def step_s0():
            layer.prepare_stacked(gu_all, dn_all, stream=stream)
            step()
        s0_total, _ = timed(step_s0, args.steps)
        with_s0 = {"ms_per_step": round(s0_total / args.steps, 4),
                   "tokens_per_s": round(tokens * args.steps / (s0_total / 1e3), 1)}

    # e2e: the public API with host buffers, copies inside the timed region.
    # Two sets of device buffers: while step i computes on `stream`, a copy
    # stream uploads step i+1's inputs and downloads step i-1's results (as a
    # training loop prefetching its next batch would); every step still moves
    # all of its own bytes inside the timed region.
    xh = x.cpu().pin_memory()
    lh = logits.cpu().pin_memory()
    dyh = dy.cpu().pin_memory() if bwd else None
    yh = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    dxh = torch.empty(y.shape, dtype=y.dtype).pin_memory() if bwd else None
    dlh = torch.empty((cfg["T"], cfg["E"]), dtype=torch.float32).pin_memory() if bwd else None
    cstream = torch.cuda.Stream(device=dev)
    sets = []
    for _ in range(2):
        sets.append(dict(x=torch.empty_like(x), l=torch.empty_like(logits),
                         dy=torch.empty_like(dy) if bwd else None, y=torch.empty_like(y),
                         g=layer.alloc_grads() if bwd else None,
                         up=torch.cuda.Event(), done=torch.cuda.Event(), down=torch.cuda.Event()))
    e2e_state = {"i": 0}

    def upload(bs):
        with torch.cuda.stream(cstream):
            cstream.wait_event(bs["down"])          # the set's previous results have left
            bs["x"].copy_(xh, non_blocking=True)
            bs["l"].copy_(lh, non_blocking=True)
            if bwd:
                bs["dy"].copy_(dyh, non_blocking=True)
            bs["up"].record(cstream)

    def download(bs):
        with torch.cuda.stream(cstream):
            cstream.wait_event(bs["done"])
            yh.copy_(bs["y"], non_blocking=True)
            if bwd:
                dxh.copy_(bs["g"]["dx"], non_blocking=True)
                dlh.copy_(bs["g"]["dlogits"], non_blocking=True)
            bs["down"].record(cstream)

    def e2e_step():
        i = e2e_state["i"]
        cur, nxt = sets[i % 2], sets[(i + 1) % 2]
        if i == 0:
            upload(cur)
        stream.wait_event(cur["up"])
        layer.forward(cur["x"], cur["l"], y=cur["y"], train=bwd, stream=stream)
        if bwd:
            layer.backward(cur["dy"], cur["x"], grads=cur["g"], stream=stream)
        cur["done"].record(stream)
        upload(nxt)                                 # overlaps this step's compute
        download(cur)
        e2e_state["i"] = i + 1

    def e2e_drain():
        stream.wait_stream(cstream)                 # the last results are on the host

    for _ in range(2):                              # warm the pipeline (not timed)
        e2e_step()
    torch.cuda.synchronize()
    e2e_state["i"] = 0

    def e2e_run():
        e2e_step()
        if e2e_state["i"] == args.steps:
            e2e_drain()

    e2e_ms, _ = timed(e2e_run, args.steps)
    h2d = x.numel() * 2 + logits.numel() * 4 + (dy.numel() * 2 if bwd else 0)
    d2h = y.numel() * 2 + ((y.numel() * 2 + cfg["T"] * cfg["E"] * 4) if bwd else 0)
    st = layer.status()
    if st != 0:
        raise RuntimeError("device status %d after the timed region" % st)

    summ = summarize(cfg, bwd, recs, args.steps, total_ms, P, write_gbs)
    mx = cfg["fmt"] == "mxfp8"
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg["fmt"],
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/d)/N(0,1/m) bf16 weights, fp32 logits)",
        "config": workload_desc(cfg, bwd, layer),
        "fwd_tokens_per_s": round(fwd_value, 1),
        "layer_roofline": layer_roofline(cfg, passes, total_ms / args.steps, P),
        "roofline": summ["roofline"],
        "kernels": summ["kernels"],
        "route_schedule_share": summ["route_schedule_share"],
        "s0_ms": round(s0_ms, 3),
        "step_with_s0": with_s0,
        "cuda_graph": graph_info,
        "e2e": {"value": round(tokens * args.steps / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": summ["gpu_launches"],
        "clocks": clk,
        "mxfp8_peak_probe": mxp,
    }
    if want_cpu:
        out["cpu_baseline"] = cpu_baseline(cfg, passes, sample, sample256, n_tok, dw_sample)
    return out, P


def cpu_baseline(cfg, passes, sample, sample256, n_tok, dw_sample=None):
    """The oracle as it stands on the host cores: the bounded n_tok-token step
    (the bench's metric, repeated to about 10 s) with BLAS on all cores and
    again on one thread, the 256-token seeded forward subset once, and (fwd+bwd)
    the weight gradients of 4 seeded experts over all their rows once."""
    cores = os.cpu_count()

    def repeat(experts):
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle_step(cfg, passes, sample, experts)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= 10.0 or reps >= 1000:
                return reps, dt

    experts, prep_s = oracle_prepare(cfg, sample)
    reps, dt = repeat(experts)
    res = {"value": round(n_tok * reps / dt, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "sample": oracle_sample_desc(cfg, passes, n_tok, len(sample["need"])) +
           "; run %d times back to back with BLAS threads = all %d cores" % (reps, cores),
           "seconds": round(dt, 2), "s0_seconds": round(prep_s, 2)}
    prev = blas_threads(1)
    if prev is not None:
        reps1, dt1 = repeat(experts)
        blas_threads(prev)
        res["one_thread"] = {"value": round(n_tok * reps1 / dt1, 4), "unit": "tokens/s", "cores": 1,
                             "seconds": round(dt1, 2), "runs": reps1}
    else:
        res["one_thread"] = {"unavailable": "no OpenBLAS thread setter found in numpy's libraries"}
    del experts
    if sample256 is not None:
        from oracle import moe as om
        ex256, prep256 = oracle_prepare(cfg, sample256)
        t0 = time.perf_counter()
        om.forward(sample256["x"], sample256["logits"], ex256, cfg["k"], cfg["fmt"], shared=sample256["shared"])
        dt = time.perf_counter() - t0
        res["fwd_256"] = {"value": round(256 / dt, 4), "unit": "tokens/s (forward)", "cores": cores,
                          "seconds": round(dt, 2), "s0_seconds": round(prep256, 2),
                          "sample": oracle_sample_desc(cfg, "fwd", 256, len(sample256["need"])) + "; run once"}
    if dw_sample is not None and dw_sample["rows"]:
        try:
            res["dw_experts"] = oracle_dw_time(cfg, dw_sample, cores)
        except Exception as exc:  # a reported baseline only: never lose the line over it
            res["dw_experts"] = {"unavailable": "%s: %s" % (type(exc).__name__, str(exc)[:160])}
    return res


def oracle_dw_time(cfg, dw_sample, cores):
    """The oracle's expert forward + backward (with dW) over every row of the
    sampled experts, once, after its own S0 for them."""
    from oracle import moe as om
    rows = dw_sample["rows"]
    exw, prepw = oracle_prepare(cfg, dw_sample)
    t0 = time.perf_counter()
    for e, (X, dY, w) in rows.items():
        W_gu, W_dn, ops = exw[e]
        fw = om.expert_forward(X, W_gu, W_dn, cfg["fmt"], ops)
        dO = om._rnd(cfg["fmt"])(w[:, None] * dY)
        om.expert_backward(dO, X, fw["GU_saved"], fw["h_saved"], W_gu, W_dn, cfg["fmt"], ops)
    dt = time.perf_counter() - t0
    n_rows = int(sum(r[0].shape[0] for r in rows.values()))
    return {"value": round(n_rows / dt, 2), "unit": "expert rows/s (forward + backward with dW)",
            "cores": cores, "seconds": round(dt, 2), "s0_seconds": round(prepw, 2),
            "sample": "%d seeded experts (%s) over all their rows (%d rows; experts with 1..2048 rows), "
                      "float64 NumPy, run once" % (len(rows), ", ".join(str(e) for e in rows), n_rows)}


def run_reference(args, cfg, passes):
    """The oracle as it stands, on the host cores, one bounded sample per step."""
    import torch
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    import moe_inputs as mi
    x = mi.tokens(cfg, dev)
    logits = mi.logits(cfg, dev)
    dy = mi.out_grad(cfg, dev) if passes == "fwdbwd" else None
    n_tok = 1 if passes == "fwdbwd" else 4
    sample = oracle_sample(cfg, passes, x, logits, dy, n_tok)
    del x, logits, dy
    experts, prep_s = oracle_prepare(cfg, sample)
    from oracle import moe as om
    for _ in range(args.warmup):          # warm-up: the routing of the sample only
        om.route(sample["logits"], cfg["k"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(cfg, passes, sample, experts)
    dt = time.perf_counter() - t0
    value = n_tok * args.steps / dt
    cores = os.cpu_count()
    return {"metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_desc(cfg, passes == "fwdbwd"),
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": oracle_sample_desc(cfg, passes, n_tok, len(sample["need"])) +
                             "; warm-up steps route the sample only", "s0_seconds": round(prep_s, 2)},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="kimi-k2.7")
    ap.add_argument("--pass", dest="passes", choices=["fwd", "fwdbwd"], default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-target", action="store_true",
                    help="skip the target leg (the MXFP8 forward of the largest workload)")
    ap.add_argument("--profile-run", action="store_true",
                    help="time the step once (no fwd-only, e2e or CPU legs): for profiler launch lists")
    ap.add_argument("--ring", type=int, default=0,
                    help="MXFP8: dispatch through a ring of this many rows (0 = materialised dispatch)")
    ap.add_argument("--gather-sms", type=int, default=0, help="gather SMs of the ring launch (0 = default)")
    ap.add_argument("--experts", choices=["bf16", "mxfp8", "nvfp4"], default=None,
                    help="the routed experts' format (default: the workload's own); nvfp4 is forward only")
    ap.add_argument("--override", default="",
                    help="comma-separated shape overrides, e.g. T=2048,E=16 (smaller cases for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    cfg = workload(args.workload)
    for kv in filter(None, args.override.split(",")):
        key, val = kv.split("=")
        cfg[key] = int(val)
    if args.experts:
        cfg["fmt"] = args.experts
        if args.experts == "nvfp4":
            cfg["backward"] = False
    passes = args.passes or ("fwdbwd" if cfg["backward"] else "fwd")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # the oracle on the host cores: rank 0 alone runs it
        if rank == 0:
            print(json.dumps(run_reference(args, cfg, passes)), flush=True)
        return
    if args.gpus != 1 or world != 1:
        ap.error("the layer runs on one GPU (no sharding, no exchange step): --gpus must be 1 and "
                 "WORLD_SIZE unset or 1 (got --gpus %d, WORLD_SIZE=%d)" % (args.gpus, world))

    import __graft_entry__
    __graft_entry__.build()
    out, P = run_ours(args, cfg, passes)
    if not (args.no_target or args.profile_run or args.override or cfg["name"] == TARGET):
        import gc
        import torch
        gc.collect()
        torch.cuda.empty_cache()
        out["target"] = run_target(args, P)
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
