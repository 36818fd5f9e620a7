"""Host-side logic of bench.py that decides what a bench line reports: the
clock record taken during the timed region (throttle reasons that reject a
run must show up), the roofline denominators, and the step's algorithmic
FLOPs.  CPU only."""
import json
import os

import numpy as np
import pytest

import bench
from precision_moe_adapter_gb300 import inputs as gi

ROW = "0, {sm}, 2070, 900.0, 0x0, {hw}, {hwt}, {swt}, {cap}"


def sampler_with(lines):
    s = bench.ClockSampler(0)
    s.out = "\n".join(lines)
    return s.summary()


def test_clock_summary_median_and_power_cap():
    na = "Not Active"
    got = sampler_with([ROW.format(sm=2070, hw=na, hwt=na, swt=na, cap=na),
                        ROW.format(sm=1980, hw=na, hwt=na, swt=na, cap="Active"),
                        ROW.format(sm=2055, hw=na, hwt=na, swt=na, cap=na)])
    assert got == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}


@pytest.mark.parametrize("which", ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"])
def test_clock_summary_reports_rejecting_reasons(which):
    flags = {k: "Not Active" for k in ("hw", "hwt", "swt", "cap")}
    flags[{"hw_slowdown": "hw", "hw_thermal_slowdown": "hwt", "sw_thermal_slowdown": "swt"}[which]] = "Active"
    got = sampler_with([ROW.format(sm=1500, **flags), "garbled line", ""])
    assert got["reasons"] == [which] and got["samples"] == 1


def test_clock_summary_without_samples():
    assert sampler_with([])["reasons"] == ["unavailable"]
    assert sampler_with(["0, N/A, N/A, N/A, N/A, N/A, N/A, N/A, N/A"])["samples"] == 0


def test_peaks_measured_and_fallback(tmp_path, monkeypatch):
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        p = bench.peaks()
        assert p["src"] == "measured" and p["hbm"] == m["hbm_gbs"]
        assert p["bf16_sus"] == m.get("bf16_tflops_sustained", m["bf16_tflops"])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def test_step_flops_of_the_kimi_workload():
    """Three expert contractions of 2*d*I per pair forward and three
    backward, the two rotations (2*dim*b per pair; four in the backward,
    the data and the adapter-gradient product), and the router."""
    cfg = gi.CONFIGS["kimi_k2"]
    fwd, bwd = bench.flops_of(cfg, cfg.P)
    assert cfg.P == cfg.T * cfg.k == 65536
    assert round((fwd + bwd) / 1e12, 2) == 11.82
    assert fwd - bwd == 2 * cfg.T * cfg.d * cfg.E - 2 * (cfg.d + cfg.I) * cfg.b * cfg.P


def test_step_bytes_count_only_active_experts():
    cfg = gi.CONFIGS["kimi_k2"]
    counts = np.zeros(cfg.E, dtype=np.int64)
    counts[:10] = 1
    b10 = bench.bytes_of(cfg, counts)
    counts[:20] = 1
    b20 = bench.bytes_of(cfg, counts)
    per_expert = (b20 - b10) / 10
    d, I = cfg.d, cfg.I
    packed = 3 * d * I // 2 + 3 * d * (I // 32) * 2       # INT4 codes + BF16 scales
    adapters = (d + I) * cfg.b * 2
    assert per_expert == 2 * (packed + adapters)         # read once in each pass


def test_peak_choice_burst_or_sustained():
    """Burst BF16 peak for a timed region at the maximum SM clock without a
    power cap; sustained otherwise (capped, or clocks well below maximum)."""
    pk = dict(hbm=6788.3, bf16=1893.4, bf16_sus=1702.3, src="measured")
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 9}
    assert bench.pick_peak(pk, full)[0] == 1893.4
    assert bench.pick_peak(pk, dict(full, reasons=["sw_power_cap"]))[0] == 1702.3
    assert bench.pick_peak(pk, dict(full, sm_mhz=1500.0))[0] == 1702.3
    assert bench.pick_peak(pk, {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]})[0] == 1702.3


def test_traffic_follows_the_gemm_sources(monkeypatch):
    """The captured DRAM traffic is reported only while the GEMM sources
    are the ones it was captured with."""
    monkeypatch.setattr(bench, "TRAFFIC", {"digest": bench.gemm_digest(),
                                           "bytes": {("kimi_k2", "fused", "gemm_gate_up"): 1e9}})
    assert bench.traffic_of("kimi_k2", "fused", "gemm_gate_up", True) == 1e9
    assert bench.traffic_of("kimi_k2", "fused", "gemm_gate_up", False) is None
    monkeypatch.setattr(bench, "TRAFFIC", {"digest": "0" * 16,
                                           "bytes": {("kimi_k2", "fused", "gemm_gate_up"): 1e9}})
    assert bench.traffic_of("kimi_k2", "fused", "gemm_gate_up", True) is None
