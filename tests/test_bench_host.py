"""Host logic of bench.py on CPU: the FLOP and byte model, the profile lookup
behind `roofline.traffic`, and the two clock samplers' summaries."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from moe_expert_ffn_route_gb300 import synth  # noqa: E402


def test_flop_model_closed_form():
    # MegaMoE notes, "performance metrics": 2 N H (2I) for L1 plus 2 N I H for L2
    wl = synth.WORKLOADS["prefill"]
    a = bench.algorithmic(wl, np.full(wl.E, wl.N // wl.E))
    N, H, I = wl.T * wl.k, wl.H, wl.I
    assert a["l1_flops"] == 2.0 * N * H * 2 * I
    assert a["l2_flops"] == 2.0 * N * I * H
    assert a["flops"] == pytest.approx(5.77e12, rel=2e-3)     # printed to three digits
    assert a["touched"] == wl.E


def test_byte_model_counts_only_touched_experts():
    wl = synth.WORKLOADS["decode"]
    counts = np.zeros(wl.E, dtype=np.int64)
    counts[:100] = 1
    a = bench.algorithmic(wl, counts)
    full = bench.algorithmic(wl, np.ones(wl.E, dtype=np.int64))
    w_per_expert = 3 * wl.I * wl.H * (0.5 + 1 / 32)       # W1 (2I x H) and W2 (H x I), E2M1 + UE8M0
    assert a["touched"] == 100
    assert full["bytes"] - a["bytes"] == pytest.approx((wl.E - 100) * w_per_expert)
    # activations: x rows in, H rows out and in again, Y rows out
    N, H, I = wl.N, wl.H, wl.I
    act = N * H * (1 + 1 / 32) + 2 * N * I * (1 + 1 / 32) + 2.0 * N * H
    assert a["bytes"] == pytest.approx(100 * w_per_expert + act)
    assert a["l1_bytes"] + a["l2_bytes"] == pytest.approx(a["bytes"])


def test_medium_step_model_matches_the_table():
    # all 64 experts touched: 6.18e11 FLOP and 8.97e8 B (roofline table of the workloads)
    wl = synth.WORKLOADS["medium"]
    a = bench.algorithmic(wl, np.ones(wl.E, dtype=np.int64))
    assert a["flops"] == pytest.approx(6.18e11, rel=2e-3)
    assert a["bytes"] == pytest.approx(8.97e8, rel=2e-3)


def test_roofline_peaks():
    pk = dict(hbm_gbs=6000.0, fp8_tflops=4000.0, fp8_tflops_sustained=3000.0, source="test")
    # prefill: tensor-bound, against the sustained FP8-rate peak, burst fraction beside it
    wl = synth.WORKLOADS["prefill"]
    a = bench.algorithmic(wl, np.full(wl.E, wl.N // wl.E))
    r = bench.gemm_roofline(a, 2.0, pk)
    tf = (a["l1_flops"] + a["l2_flops"]) / 2e-3 / 1e12
    assert r["bound"] == "tensor" and r["peak"] == 3000.0
    assert r["frac"] == pytest.approx(tf / 3000.0) and r["frac_of_burst_peak"] == pytest.approx(tf / 4000.0)
    assert bench.step_roofline_time(a, pk) == pytest.approx(a["flops"] / 4e15)
    assert bench.step_roofline_time(a, pk, True) == pytest.approx(a["flops"] / 3e15)
    # decode: weight streaming, against the HBM copy bandwidth
    wl = synth.WORKLOADS["decode"]
    a = bench.algorithmic(wl, np.ones(wl.E, dtype=np.int64))
    r = bench.gemm_roofline(a, 1.0, pk)
    assert r["bound"] == "hbm" and r["peak"] == 6000.0 and "frac_of_burst_peak" not in r
    assert r["frac"] == pytest.approx((a["l1_bytes"] + a["l2_bytes"]) / 1e-3 / 1e9 / 6000.0)


def test_traffic_lookup_follows_the_kernel_hash():
    text = open(os.path.join(ROOT, "profiles", "grouped_gemm_traffic.md")).read()
    recorded = text.split("kernel source sha256:")[1].split()[0]
    assert bench.traffic_from_profile(recorded, "prefill", 1.0) == 7550064640.0
    assert bench.traffic_from_profile(recorded, "prefill", 2.0) == 2 * 7550064640.0
    assert bench.traffic_from_profile(recorded, "decode", 1.0) == 6010465480.0
    assert bench.traffic_from_profile("0" * 64, "prefill", 1.0) is None     # another kernel source
    assert bench.traffic_from_profile(recorded, "no-such-workload", 1.0) is None


def test_kernel_hash_is_stable():
    h = bench.kernel_hash()
    assert len(h) == 64 and h == bench.kernel_hash()


def test_nvidia_smi_summary():
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1995, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1201.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
    ]
    got = s.summary()
    assert got["samples"] == 3 and got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]


def test_nvml_summary_decodes_reason_bits():
    s = object.__new__(bench.NvmlSampler)          # no NVML here: fill the record by hand
    s.max_mhz = 2070.0
    s.samples = [(2070.0, 0x0), (1800.0, 0x4 | 0x1), (1500.0, 0x40), (2070.0, 0x8 | 0x20)]
    got = s.summary()
    assert got["samples"] == 4 and got["sm_mhz"] == pytest.approx(1935.0)
    assert got["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    s.samples = []
    assert s.summary()["sm_mhz"] is None


def test_clock_sampler_falls_back_without_nvml(monkeypatch):
    class Dev:
        index = 0

    def no_nvml(dev):
        raise OSError("no NVML")

    monkeypatch.setattr(bench, "NvmlSampler", no_nvml)
    assert isinstance(bench.clock_sampler(Dev()), bench.ClockSampler)
