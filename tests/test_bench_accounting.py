"""Host arithmetic behind the bench's roofline figures, on CPU.

The layer figures are pinned to numbers worked out by hand from the layer
shapes (6·d·m FLOPs per routed (token, expert) pair plus 6·d·m_s per token for
the shared expert; weights once in their stored format plus the layer-boundary
activations), written here to three significant figures.  The per-kernel work
is pinned by invariants: the expert GEMMs of one pass add up to the layer's
FLOPs, and the backward's four GEMMs are twice the forward's two."""
import os

import pytest

import bench

# (FLOPs fwd, algorithmic GB fwd, GB fwd+bwd or None)
HAND = {
    "qwen3.5-397b": (2.27e12, 13.06, None),
    "glm-5.2": (9.90e12, 10.39, None),
    "kimi-k2.7": (1.30e13, 18.0, 70.0),
    "deepseek-v4-pro": (2.60e13, 27.15, None),
}


@pytest.mark.parametrize("name", list(HAND))
def test_layer_work_matches_hand_figures(name):
    cfg = bench.workload(name)
    flops, gb, gb_bwd = HAND[name]
    f, fs, b = bench.layer_work(cfg, "fwd")
    assert f + fs == pytest.approx(flops, rel=5e-3)
    assert b / 1e9 == pytest.approx(gb, rel=5e-3)
    if gb_bwd is not None:
        f3, fs3, b3 = bench.layer_work(cfg, "fwdbwd")
        assert f3 + fs3 == pytest.approx(3 * (f + fs))
        assert b3 / 1e9 == pytest.approx(gb_bwd, rel=5e-3)


FWD = ("gemm1_gate_up_swiglu", "gemm2_down")
BWD = ("dgrad_down_swiglu_bwd", "dgrad_gate_up", "wgrad_down", "wgrad_gate_up")


@pytest.mark.parametrize("name", ["tiny", "kimi-k2.7", "deepseek-v4-pro"])
def test_kernel_flops_add_up_to_the_layer(name):
    cfg = bench.workload(name)
    fl_exp, fl_sh, _ = bench.layer_work(cfg, "fwd")
    fwd = sum(bench.kernel_work(cfg, n, False)[0] for n in FWD)
    bwd = sum(bench.kernel_work(cfg, n, True)[0] for n in BWD)
    assert fwd == pytest.approx(fl_exp)
    assert bwd == pytest.approx(2 * fl_exp)
    if cfg["m_shared"]:
        sh = sum(bench.kernel_work(cfg, "shared_" + n, False)[0] for n in FWD)
        sh_b = sum(bench.kernel_work(cfg, "shared_" + n, True)[0] for n in BWD)
        assert sh == pytest.approx(fl_sh)
        assert sh_b == pytest.approx(2 * fl_sh)


def test_kernel_roofline_takes_the_longer_bound():
    cfg = bench.workload("kimi-k2.7")
    measured = {"hbm_gbs": 6757.9, "bf16_tflops": 1856.7, "bf16_tflops_sustained": 1661.6}
    peaks = bench.tensor_peaks(measured, "measured", {"burst_tflops": 3771.5, "sustained_tflops": 3400.0,
                                                      "how": "test"})
    # the gate/up wgrad writes 22.5 GB of bf16 dW: HBM-bound at this shape
    r = bench.kernel_roofline(cfg, "wgrad_gate_up", True, 6.0, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    byts = bench.kernel_work(cfg, "wgrad_gate_up", True)[1]
    assert r["achieved"] == pytest.approx(byts / 6.0e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6757.9)
    assert r["frac_nominal"] == pytest.approx(r["achieved"] / bench.NOMINAL["hbm_gbs"])
    # the forward gate/up GEMM is tensor-bound, at the measured MXFP8 rate
    r = bench.kernel_roofline(cfg, "gemm1_gate_up_swiglu", False, 3.6, peaks)
    assert r["bound"] == "tensor" and r["mx"]
    assert r["peak"] == pytest.approx(3771.5)
    assert r["frac_sustained"] == pytest.approx(r["achieved"] / 3400.0)
    assert r["frac_nominal"] == pytest.approx(r["achieved"] / 4500.0)
    # a BF16 GEMM (shared expert) against the burst BF16 rate
    r = bench.kernel_roofline(cfg, "shared_gemm2_down", False, 0.25, peaks)
    assert r["bound"] == "tensor" and not r["mx"] and r["peak"] == pytest.approx(1856.7)
    # without the MXFP8 probe the ratio of the measured BF16 rates stands in, labelled so
    fb = bench.tensor_peaks(measured, "measured", {"burst_tflops": None})
    assert fb["mx"] == pytest.approx(2 * 1856.7) and "unavailable" in fb["mx_src"]


def test_layer_roofline_fractions():
    cfg = bench.workload("deepseek-v4-pro")
    peaks = bench.tensor_peaks({"hbm_gbs": 6757.9, "bf16_tflops": 1856.7, "bf16_tflops_sustained": 1661.6},
                               "measured", {"burst_tflops": 3771.5, "sustained_tflops": 3400.0, "how": "test"})
    fl_exp, fl_sh, byt = bench.layer_work(cfg, "fwd")
    t_roof = max(fl_exp / 3771.5e12, byt / 6757.9e9)
    lr = bench.layer_roofline(cfg, "fwd", 12.0, peaks)
    assert lr["bound"] == "tensor"
    assert lr["frac"] == pytest.approx(t_roof / 12.0e-3, abs=1e-4)
    assert lr["frac_nominal"] == pytest.approx(max(fl_exp / 4500e12, byt / 7900e9) / 12.0e-3, abs=1e-4)
    cfg = bench.workload("kimi-k2.7")
    assert bench.kernel_roofline(cfg, "no_such_kernel", True, 1.0, peaks) is None


def test_launches_per_traced_region():
    mx = bench.workload("kimi-k2.7")
    bf = bench.workload("qwen3.5-397b")
    assert bench.kernels_in_region("route_schedule", mx, True) == 4
    assert bench.kernels_in_region("dispatch_gather", mx, True) == 2
    assert bench.kernels_in_region("dispatch_gather", mx, False) == 3
    assert bench.kernels_in_region("dispatch_gather", bf, False) == 1
    assert bench.kernels_in_region("wgrad_gate_up", mx, True) == 2
    assert bench.kernels_in_region("gemm1_gate_up_swiglu", mx, True) == 1


def _experts_with_rows(wl):
    """Experts the workload's routing gives rows to, from the oracle's top-k of
    logits drawn on the CPU (the bench draws the same distribution on the GPU,
    where the count comes out a few experts higher: 232 against 225 for
    Kimi-K2.7); close enough for the bounds below."""
    import numpy as np
    import torch
    import moe_inputs as mi
    from oracle import moe as om
    cfg = dict(mi.WORKLOADS[wl])
    idx, _ = om.route(mi.logits(cfg, torch.device("cpu")).numpy(), cfg["k"])
    return int((np.bincount(idx.reshape(-1), minlength=cfg["E"]) > 0).sum())


def test_recorded_traffic_names_a_known_kernel():
    active = {}
    for (wl, kernel), traffic in bench.NCU_TRAFFIC.items():
        cfg = bench.workload(wl)
        if wl not in active:
            active[wl] = _experts_with_rows(wl)
        cfg["E_active"] = active[wl]
        w = bench.kernel_work(cfg, kernel, cfg["backward"])
        assert w is not None
        # DRAM traffic of a full-size launch: at least the algorithmic bytes
        # (less only by what L2 still holds at the end), and not wildly above
        assert 0.95 * w[1] < traffic < 1.5 * w[1], (wl, kernel, traffic / w[1])


def test_only_experts_with_rows_count_as_weight_reads():
    """An empty expert's weights are never read; its dW is still written."""
    cfg = bench.workload("kimi-k2.7")
    full = {n: bench.kernel_work(cfg, n, True)[1] for n in ("gemm2_down", "wgrad_down")}
    cfg["E_active"] = cfg["E"] - 100
    part = {n: bench.kernel_work(cfg, n, True)[1] for n in ("gemm2_down", "wgrad_down")}
    w = 100 * cfg["d"] * cfg["m"] * bench.elem_bytes(cfg)
    assert full["gemm2_down"] - part["gemm2_down"] == pytest.approx(w)
    assert full["wgrad_down"] == part["wgrad_down"]
    fwd = bench.layer_work(cfg, "fwd")[2]
    cfg.pop("E_active")
    assert bench.layer_work(cfg, "fwd")[2] - fwd == pytest.approx(3 * w)


def test_clock_records_that_reject_a_number():
    ok = {"sm_mhz": 2040.0, "sm_max_mhz": 2070.0, "reasons": []}
    capped = {"sm_mhz": 1950.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    thermal = {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["hw_thermal_slowdown", "sw_power_cap"]}
    locked = {"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": []}
    low_capped = {"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    unknown = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(capped)
    assert bench.clocks_rejected(thermal)
    assert bench.clocks_rejected(locked)
    assert not bench.clocks_rejected(low_capped)
    assert not bench.clocks_rejected(unknown)


def test_clock_sampler_against_a_fake_nvidia_smi(tmp_path, monkeypatch):
    """The sampler waits for the first sample, then parses the query's CSV
    (index, sm, max sm, power, active, four reason columns)."""
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "i=0\n"
                    "while [ $i -lt 50 ]; do\n"
                    "  echo '0, 1980, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "  i=$((i+1)); sleep 0.05\n"
                    "done\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", str(tmp_path) + os.pathsep + os.environ["PATH"])
    clk = bench.Clocks(0)
    assert os.path.getsize(clk.f.name) > 0          # a sample was on file before timing
    rec = clk.stop()
    assert rec["sm_mhz"] == 1980.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"] and rec["samples"] >= 1
    assert not bench.clocks_rejected(rec)


def test_dw_sample_takes_every_row_of_seeded_small_experts():
    """The CPU baseline's weight-gradient leg: 4 seeded experts with 1..max_rows
    rows, each with exactly the tokens and combine weights routed to it."""
    import numpy as np
    import torch

    T, k, E = 64, 2, 8
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[:, 0] = np.where(np.arange(T) < 40, 0, idx[:, 0])    # expert 0 gets many rows
    idx[:, 1] = np.where(idx[:, 1] == idx[:, 0], (idx[:, 0] + 1) % E, idx[:, 1])
    w = rng.random((T, k)).astype(np.float32)
    counts = np.bincount(idx.reshape(-1), minlength=E).astype(np.int32)

    class FakeLayer:
        def view(self, which, name, dtype, shape):
            assert which == 0
            return torch.as_tensor({"counts": counts, "idx": idx, "w": w}[name]).reshape(shape)

    cfg = dict(T=T, d=64, m=32, E=E, k=k, m_shared=0, fmt="bf16", bias="none", seed=9, backward=True)
    x = torch.randn(T, cfg["d"]).to(torch.bfloat16)
    dy = torch.randn(T, cfg["d"]).to(torch.bfloat16)
    s = bench.oracle_dw_sample(cfg, FakeLayer(), x, dy, n=4, max_rows=30)
    assert len(s["rows"]) == 4 and 0 not in s["rows"]          # expert 0 (40+ rows) is over the cap
    for e, (X, dY, we) in s["rows"].items():
        slots = np.nonzero(idx.reshape(-1) == e)[0]
        assert 1 <= slots.size <= 30 and X.shape == (slots.size, cfg["d"])
        assert np.array_equal(X, x[slots // k].float().numpy().astype(np.float64))
        assert np.array_equal(dY, dy[slots // k].float().numpy().astype(np.float64))
        assert np.array_equal(we, w.reshape(-1)[slots].astype(np.float64))
        assert s["masters"][e][0].shape == (2 * cfg["m"], cfg["d"])
