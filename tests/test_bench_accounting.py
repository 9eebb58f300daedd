"""The measurement arithmetic of bench.py, on the CPU: the roofline peaks
derived from the measured rates, the FLOP count of an attention call, the
algorithmic bytes of the group and prep steps, and the DRAM traffic taken
from the committed ncu record (scaled by B*H*N, withheld once the kernel's
sources change)."""
import importlib.util
import json
import os

import pytest

from bit_attention_video_smooth_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_attention_flops_of_the_wan_call():
    w = I.WORKLOADS["wan"]
    assert w.flops == 4 * w.B * w.H * w.N * w.N * 128
    assert abs(w.flops / 1e12 - 102.24) < 0.01


def test_peaks_from_the_measured_rates(bench):
    """The attention kernels run at full clock without the power cap: their
    peaks come from the burst cuBLAS bf16 rate b (FP8 = 2 b by the nominal
    ratio 4.5 / 2.25), never from the power-capped sustained figure."""
    peaks = {"bf16_tflops": 1950.6, "bf16_tflops_sustained": 1717.9}
    fp8, src = bench.attention_peak("e4m3", peaks)
    assert fp8 == pytest.approx(3901.2) and "burst" in src
    fp4, _ = bench.attention_peak("nvfp4", peaks)
    # QK at the FP8 rate (2b), PV as the block-scaled FP4 MMA at 6b: 1 / (0.5 / 2b + 0.5 / 6b)
    assert fp4 == pytest.approx(1.0 / (0.5 / 3901.2 + 0.5 / (6 * 1950.6)))
    fallback, src = bench.attention_peak("e4m3", None)
    assert fallback == pytest.approx(3800.0) and "fallback" in src
    # against nominal dense rates: FP8 4.5 PF; the NVFP4 kernel's QK at FP8, PV at FP4 13.5 PF
    assert bench.attention_nominal("e4m3") == pytest.approx(4500.0)
    assert bench.attention_nominal("nvfp4") == pytest.approx(1.0 / (0.5 / 4500.0 + 0.5 / 13500.0))


def test_algorithmic_bytes(bench):
    w = I.WORKLOADS["wan"]
    # eight rounds of (V read, labels written) plus the sort's labels and permutation
    assert bench.group_bytes(w) == pytest.approx(8 * 40 * 70656 * (256 + 4) + 40 * 70656 * 8)
    assert bench.group_bytes(w) / 1e9 == pytest.approx(5.90, abs=0.01)
    # Q, K, V and perm read; q8, k8, v_res written; means, block scales, channel scales
    nb = 70656 // 128
    assert bench.prep_bytes(w) == pytest.approx(40 * (70656 * (768 + 4 + 256 + 128) + nb * (256 + 8) + 512))
    assert bench.prep_bytes(w) / 1e9 == pytest.approx(3.27, abs=0.01)
    w4 = I.WORKLOADS["nvfp4"]
    # NVFP4 residual: 64 bytes of codes and 8 scales per token instead of 128 bytes
    assert bench.prep_bytes(w4) < bench.prep_bytes(I.with_n(w, w4.N, H=w4.BH))


def test_traffic_scales_with_the_work_and_tracks_the_sources(bench, monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "attention_traffic.json")))["attention_e4m3_kernel"]
    w = I.WORKLOADS["wan"]
    c = rec["captured_on"]
    expect = rec["dram_bytes_per_launch"] * (w.B * w.H * w.N) / (c["B"] * c["H"] * c["N"])
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda files: rec["sources_sha256"])
    assert bench.attention_traffic(w) == pytest.approx(expect)
    # a capture of other sources is not reported
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda files: "0" * 64)
    assert bench.attention_traffic(w) is None


def test_clock_sampler_names_the_device_nvidia_smi_sees(bench, monkeypatch):
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES", raising=False)
    assert bench.ClockSampler.smi_id(0) == "0"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "5,2")
    assert bench.ClockSampler.smi_id(0) == "5" and bench.ClockSampler.smi_id(1) == "2"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-8f0c, 3")
    assert bench.ClockSampler.smi_id(0) == "GPU-8f0c" and bench.ClockSampler.smi_id(1) == "3"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "")
    assert bench.ClockSampler.smi_id(0) == "0"


def test_clock_summary_reasons_and_median(bench):
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1950, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 2010, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "garbage line"]
    s = c.summary()
    assert s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    c.lines = []
    assert c.summary()["reasons"] == ["unsampled"]
