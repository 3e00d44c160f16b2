"""Host-side pieces of bench.py that decide whether a measurement stands: the
clock summary taken during the timed region (from nvidia-smi lines, faked
here) and the DRAM-traffic record, which counts only while the kernel source
is the one the counters were taken from."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _line(sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return f"0, {sm}, {mx}, 900.0, 0x0, {hw}, {hwt}, {swt}, {cap}"


def test_clock_summary_of_a_clean_run():
    lines = [_line(2070, 2070)] * 5 + [_line(600, 2070)]  # one idle sample, left out of the median
    c = bench.ClockSampler.summarize(lines)
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070 and c["reasons"] == [] and c["samples"] == 6


def test_clock_summary_reports_throttle_reasons():
    lines = [_line(2070, 2070), _line(1800, 2070, hw="Active"), _line(1900, 2070, cap="Active"),
             _line(1950, 2070, hwt="Active", swt="Active")]
    c = bench.ClockSampler.summarize(lines)
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert c["sm_mhz"] == pytest.approx(1925.0)


def test_clock_summary_skips_malformed_lines():
    c = bench.ClockSampler.summarize(["", "garbage", "0, [N/A], 2070, 1, 2, 3, 4, 5, 6"])
    assert c["sm_mhz"] is None and c["reasons"] == ["no samples"]


def test_traffic_record_counts_only_for_the_profiled_source(tmp_path, monkeypatch):
    src = tmp_path / "quantized_moe_expert_top_gb300" / "csrc"
    src.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (src / "gemm_pair.cu").write_bytes(b"// kernel v1\n")
    sha = hashlib.sha256(b"// kernel v1\n").hexdigest()[:16]
    rel = "quantized_moe_expert_top_gb300/csrc/gemm_pair.cu"
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps({"records": [
        {"kernel": "gemm_gateup", "workload": "prefill", "source": rel, "source_sha256_16": sha,
         "bytes_per_launch": 123},
        {"kernel": "gemm_down", "workload": "prefill", "source": rel, "source_sha256_16": sha,
         "bytes_per_launch": 45}]}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("gemm_gateup", "prefill") == 123
    assert bench.measured_traffic("gemm_down", "prefill") == 45
    assert bench.measured_traffic("gemm_down", "decode1") is None   # no record for that workload
    assert bench.measured_traffic("act_quant", "prefill") is None
    (src / "gemm_pair.cu").write_bytes(b"// kernel v2\n")  # changed since the capture
    assert bench.measured_traffic("gemm_gateup", "prefill") is None


def test_algorithmic_bytes_follow_the_layer_not_the_implementation():
    import synth
    wl = synth.WORKLOADS["prefill"]
    counts = [wl.T * wl.k // wl.E] * wl.E
    import numpy as np
    acc = bench.workload_accounting(wl, np.array(counts))
    # gate/up: 256 experts x 2 x 2048 x 4096 x 17/32 B of weights + x in bf16
    assert acc["gemm_gateup_bytes"] == 256 * 2 * 2048 * 4096 * 17 // 32 + 4096 * 4096 * 2
    # down: weights + out in fp32; the MXFP8 rows are implementation bytes
    assert acc["gemm_down_bytes"] == 256 * 4096 * 2048 * 17 // 32 + 4096 * 4096 * 4
    assert acc["implementation_bytes"]["gemm_gateup"] == 32768 * (4096 + 2048) * 33 // 32
    assert acc["total_bytes"] == 3422552064 + 4096 * 4096 * 2 + 4096 * 256 * 4 + 4096 * 4096 * 4


def test_dominant_roofline_picks_the_slowest_kernel_and_its_bound():
    """The roofline object follows the kernel with the largest live time: its
    algorithmic bytes over its time against the HBM peak, or its FLOP against
    the MXFP8 peak when those would take longer at that peak; worked by hand."""
    import numpy as np
    import synth
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "source": "measured"}
    wl = synth.WORKLOADS["decode64"]
    counts = np.zeros(wl.E, int)
    counts[:64] = 8                                   # 64 touched experts, 512 pairs
    acc = bench.workload_accounting(wl, counts)
    r = bench.dominant_roofline({"decode_mma_gateup": 0.1, "decode_mma_down": 0.05, "route_topk": 0.01},
                                acc, "no-such-workload", peaks, 4000.0, 12000.0)
    assert r["kernel"] == "decode_mma_gateup" and r["bound"] == "hbm" and r["traffic"] is None
    gate_up = 64 * 2 * wl.f * (wl.d // 2 + wl.d // 32)  # gate and up rows of 64 experts: codes + scales
    assert acc["decode_gateup_bytes"] >= gate_up
    assert r["achieved"] == pytest.approx(acc["decode_gateup_bytes"] / 0.1e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6000.0)
    # the prefill chunk's gate/up: 2.3 GB at 6 TB/s (0.39 ms) outlast 1.1 TFLOP at 4 PF (0.27 ms), so it is
    # HBM-bound; at a 2 PF tensor peak the FLOP (0.55 ms) would bound it instead
    wl = synth.WORKLOADS["prefill"]
    acc = bench.workload_accounting(wl, np.full(wl.E, wl.T * wl.k // wl.E))
    flops = 2 * wl.T * wl.k * wl.d * 2 * wl.f
    assert acc["flops_gateup"] == flops
    r = bench.dominant_roofline({"gemm_gateup": 0.5, "gemm_down": 0.3}, acc, "prefill", peaks, 4000.0, 12000.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["tensor_frac_of_mxf8f6f4_peak"] == pytest.approx(flops / 0.5e-3 / 1e12 / 4000.0)
    r = bench.dominant_roofline({"gemm_gateup": 0.5, "gemm_down": 0.3}, acc, "prefill", peaks, 2000.0, 6000.0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(flops / 0.5e-3 / 1e12)
    assert r["hbm_frac"] == pytest.approx(acc["gemm_gateup_bytes"] / 0.5e-3 / 1e9 / 6000.0)
    assert bench.dominant_roofline({}, acc, "prefill", peaks, 4000.0, 12000.0) is None


def test_config_states_the_l2_rule_of_the_timed_steps():
    """Both arms print config_of(...) unchanged; it says how L2 is kept out
    of the timing, by the same rule the timed loop follows."""
    import synth
    pre, dec = synth.WORKLOADS["prefill"], synth.WORKLOADS["decode1"]
    assert not bench.flushes_l2(pre) and bench.flushes_l2(dec)
    c = bench.config_of(pre, 1)
    # 256 experts x (gate + up MXFP4 [2048 x 4096] + down MXFP4 [4096 x 2048]) = 3.42 GB > the 129 MB L2
    assert c["l2"].startswith("inputs larger than L2") and "3.42 GB" in c["l2"]
    assert bench.config_of(dec, 1)["l2"].startswith("flushed")
    assert c["workload"].startswith("prefill: T=4096 d=4096 E=256 f=2048 top_k=8")
