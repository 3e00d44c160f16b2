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
