#!/usr/bin/env python3
"""Benchmark of the routed-MoE expert layer (MXFP4 experts) on GB300.

One step = one forward pass of the whole layer (routing, grouping, MXFP8
activation quantisation, grouped gate/up GEMM + SwiGLU, grouped down GEMM +
weighted combine) over one batch of synthetic tokens.  The default workload is
the 4096-token prefill chunk (d=4096, 256 experts, f=2048, top-8); the line
also carries the few-token decode workloads (T=1, T=64 Zipf) and the Q2_K
down-projection variant (T=2048) measured on the same GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 runs under torchrun: every rank runs an independent replica of the
layer on its own GPU (the layer has no data-path exchange); the value is the
tokens of all ranks divided by the slowest rank's time.

--impl reference times the CPU oracle (the plain fp64 C restatement used for
parity) on this host's cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s (decode T=1/64, prefill T=4096) + % HBM / FP4 roofline"


# ----------------------------------------------------------------- accounting
def mxfp4_bytes(rows: int, K: int) -> int:
    return rows * K // 2 + rows * K // 32


def q2k_bytes(rows: int, K: int) -> int:
    return rows * (K // 256) * 84


def workload_accounting(wl: synth.Workload, counts: np.ndarray) -> dict:
    """Algorithmic bytes and flops of one forward, per kernel and in total.

    Algorithmic bytes are what the layer must move: the weights of every
    touched expert once (U = experts with >= 1 token), x read once (bf16), the
    logits read once and out written once (fp32).  Per kernel: gate/up = its
    weights + x, down = its weights + out.  The MXFP8 (or fp16) activation
    rows that the grouped GEMMs exchange through HBM (x^ per routed pair, h)
    belong to this implementation, not to the layer, and are reported apart as
    implementation bytes."""
    T, d, f, k, E = wl.T, wl.d, wl.f, wl.k, wl.E
    U = int((counts > 0).sum())
    pairs = T * k
    gu_w = U * 2 * mxfp4_bytes(f, d)
    dn_w = U * (q2k_bytes(d, f) if wl.down == "q2k" else mxfp4_bytes(d, f))
    io = T * d * 2 + T * E * 4 + T * d * 4
    flops_gu = 2.0 * pairs * d * 2 * f
    flops_dn = 2.0 * pairs * f * d
    return {
        "U": U,
        "weights_gateup": gu_w,
        "weights_down": dn_w,
        "io": io,
        "total_bytes": gu_w + dn_w + io,
        # per-kernel algorithmic bytes: the kernel's weights + the layer input or output it touches
        "gemm_gateup_bytes": gu_w + T * d * 2,
        "gemm_down_bytes": dn_w + T * d * 4,
        "decode_gateup_bytes": gu_w + T * d * 2,
        "decode_down_bytes": dn_w + T * d * 4,
        # activation rows exchanged through HBM by this implementation (prefill path)
        "implementation_bytes": {
            "gemm_gateup": pairs * d * 33 // 32 + (pairs * f * 2 if wl.down == "q2k" else pairs * f * 33 // 32),
            "gemm_down": pairs * f * 2 if wl.down == "q2k" else pairs * f * 33 // 32,
        },
        "flops_gateup": flops_gu,
        "flops_down": flops_dn,
        "flops": flops_gu + flops_dn,
    }


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the
    committed ncu record (profiles/dram_traffic.json), or None when there is no
    record or the kernel's source file changed since the counters were taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as fh:
            recs = json.load(fh)["records"]
    except (OSError, ValueError, KeyError):
        return None
    for r in recs:
        if r.get("kernel") != kernel or r.get("workload") != workload:
            continue
        try:
            src = os.path.join(ROOT, r["source"])
            sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        except (OSError, KeyError):
            return None
        return r.get("bytes_per_launch") if sha == r.get("source_sha256_16") else None
    return None


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            m = json.load(fh)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summarize(self.lines)

    @staticmethod
    def summarize(lines) -> dict:
        """Median SM clock of the loaded samples (above half the highest), the
        highest max clock, and the throttle reasons seen active in any sample,
        from `nvidia-smi --format=csv,noheader,nounits` lines of FIELDS."""
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [s for s in sms if s > 0.5 * max(sms)] or sms
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(maxs), "reasons": sorted(reasons),
                "samples": len(sms)}


# ----------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    """The largest of the ranks' values (the slowest rank's step time)."""
    if ws == 1:
        return v
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(ws: int, tokens_per_rank: int, ms_step_max: float) -> float:
    """Whole-job tokens/s: every rank runs an independent replica on its own
    tokens (weak scaling), timed by the slowest rank."""
    return ws * tokens_per_rank / (ms_step_max * 1e-3)


class L2Flush:
    """Flushes L2 between timed decode steps: writes a buffer larger than L2
    (512 MB), then reads it back, so the step that follows finds L2 holding
    only clean lines of an unrelated buffer (no write-backs charged to it)."""

    def __init__(self):
        self.buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
        self.sink = torch.empty(1, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.buf.fill_(1.0)
        torch.sum(self.buf, dim=0, keepdim=True, out=self.sink)


def run_forward(layer, x, logits, out):
    """One forward: given logits, or (logits None) the whole layer from x."""
    if logits is None:
        layer.forward_x(x, out)
    else:
        layer.forward(x, logits, out)


def time_steps(layer, x, logits, out, steps, flush=None, kernel_times=False):
    """Times `steps` forwards with CUDA events on the current stream; returns
    (per-step ms list, per-kernel ms dict of lists)."""
    st = torch.cuda.current_stream()
    per_step, per_kernel = [], {}
    layer.set_kernel_timing(kernel_times)
    for _ in range(steps):
        if flush is not None:
            flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        run_forward(layer, x, logits, out)
        e1.record(st)
        e1.synchronize()
        per_step.append(e0.elapsed_time(e1))
        if kernel_times:
            for name, ms in layer.kernel_times().items():
                per_kernel.setdefault(name, []).append(ms)
    layer.set_kernel_timing(False)
    return per_step, per_kernel


def routing_counts(wl: synth.Workload, logits: torch.Tensor) -> np.ndarray:
    """Expert loads of the workload's routing (top-k of the logits; this is
    bookkeeping for the byte count only, not a result of the layer)."""
    top = torch.topk(logits.float(), wl.k, dim=1).indices.cpu().numpy()
    return np.bincount(top.ravel(), minlength=wl.E)


# ----------------------------------------------------------------- our arm
def measure_workload(ds4, layer, wl, steps, warmup, peaks, flush, want_kernels=True, with_x=False) -> dict:
    inp = synth.make_inputs(wl, device="cuda")
    x, logits = inp["x"], (None if with_x else inp["logits"])
    out = torch.empty(wl.T, wl.d, dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        if flush:
            flush()
        run_forward(layer, x, logits, out)
    torch.cuda.synchronize()
    if layer.status() != ds4.OK:
        raise RuntimeError(f"{wl.name}: device status {ds4.status_string(layer.status())}")
    per_step, _ = time_steps(layer, x, logits, out, steps, flush, kernel_times=False)
    kern = {}
    if want_kernels:
        _, kern = time_steps(layer, x, logits, out, min(steps, 20), flush, kernel_times=True)
    torch.cuda.synchronize()
    if layer.status() != ds4.OK:
        raise RuntimeError(f"{wl.name}: device status after timing")
    # the expert loads: of the given logits, or (from x) of the logits the layer's router produced
    acc = workload_accounting(wl, routing_counts(wl, logits if logits is not None else layer.logits()))
    ms = statistics.median(per_step)
    res = {"T": wl.T, "ms": ms, "tokens_per_s": wl.T / (ms * 1e-3), "U": acc["U"],
           "GBps": acc["total_bytes"] / (ms * 1e-3) / 1e9,
           "TFLOPs": acc["flops"] / (ms * 1e-3) / 1e12,
           "hbm_frac_of_measured": acc["total_bytes"] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
           "kernels_ms": {k: statistics.median(v) for k, v in kern.items()},
           "launches": layer.launches_per_forward(wl.T),
           "path": {1: "decode (CUDA-core GEMV)", 2: "prefill (MXFP8 tcgen05 GEMM)",
                    3: "decode_mma (split-precision tcgen05 GEMM)"}.get(layer.path_for(wl.T), "?")}
    return res, acc, x, logits, out


def flushes_l2(wl: synth.Workload) -> bool:
    """The decode workloads (T <= 64) read less than L2 holds: L2 is flushed
    before every timed step.  The larger ones read more than L2 per step."""
    return wl.T <= 64


def config_of(wl: synth.Workload, ws: int) -> dict:
    """The `config` object of the JSON line, identical in both arms."""
    per_expert = 2 * mxfp4_bytes(wl.f, wl.d) + (q2k_bytes(wl.d, wl.f) if wl.down == "q2k" else mxfp4_bytes(wl.d, wl.f))
    l2 = ("flushed (512 MB write + read back) before every step" if flushes_l2(wl) else
          "inputs larger than L2: the touched experts' weights, up to %.2f GB per step" % (wl.E * per_expert / 1e9))
    return {"workload": f"{wl.name}: T={wl.T} d={wl.d} E={wl.E} f={wl.f} top_k={wl.k} down={wl.down}",
            "T": wl.T, "d": wl.d, "E": wl.E, "f": wl.f, "top_k": wl.k, "routing": wl.routing,
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU", "l2": l2}


def dominant_roofline(kms: dict, acc: dict, workload: str, peaks: dict, fp8_peak: float, fp4_peak: float):
    """Roofline of the kernel with the largest live event time: its
    algorithmic bytes (or FLOP) per launch over its mean time, against the
    measured HBM peak (or the MXFP8 tensor peak when the launch's FLOP take
    longer at that peak than its bytes at the HBM peak), with the ncu DRAM
    traffic of the same launch when a current record exists."""
    dom = max(kms, key=kms.get) if kms else None
    bytes_key = {"gemm_gateup": "gemm_gateup_bytes", "gemm_down": "gemm_down_bytes",
                 "decode_mma_gateup": "decode_gateup_bytes", "decode_mma_down": "decode_down_bytes",
                 "decode_gateup": "decode_gateup_bytes", "decode_down": "decode_down_bytes"}
    flops_key = {"gemm_gateup": "flops_gateup", "gemm_down": "flops_down",
                 "decode_mma_gateup": "flops_gateup", "decode_mma_down": "flops_down",
                 "decode_gateup": "flops_gateup", "decode_down": "flops_down"}
    if dom not in bytes_key:
        return None
    t = kms[dom] * 1e-3
    gbs = acc[bytes_key[dom]] / t / 1e9
    tfl = acc[flops_key[dom]] / t / 1e12
    hbm_time = acc[bytes_key[dom]] / (peaks["hbm_gbs"] * 1e9)
    tc_time = acc[flops_key[dom]] / (fp8_peak * 1e12)
    if dom.startswith("gemm") and tc_time > hbm_time:
        roofline = {"bound": "tensor", "achieved": tfl, "peak": fp8_peak, "unit": "TFLOP/s", "frac": tfl / fp8_peak}
    else:
        roofline = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"]}
    roofline.update({"kernel": dom, "kernel_ms": kms[dom],
                     "traffic": measured_traffic(dom, workload),
                     "implementation_bytes": acc["implementation_bytes"].get(dom),
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
                     else "fallback",
                     "algorithmic_bytes": acc[bytes_key[dom]], "algorithmic_flops": acc[flops_key[dom]]})
    if dom.startswith("gemm"):
        roofline["tensor_frac_of_mxf8f6f4_peak"] = tfl / fp8_peak
        roofline["tensor_frac_of_fp4_peak"] = tfl / fp4_peak
        roofline["hbm_frac"] = gbs / peaks["hbm_gbs"]
    return roofline


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    import quantized_moe_expert_top_gb300 as ds4
    ds4.build()
    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * 2.0  # kind::mxf8f6f4 runs at the fp8 rate: nominal 4.5 / 2.25 PF
    fp4_peak = peaks["bf16_tflops"] * 6.0  # nominal 13.5 / 2.25 PF

    wl = synth.WORKLOADS[args.workload]
    base = synth.WORKLOADS["prefill"]  # one layer serves decode1 / decode64 / prefill
    # the decode and prefill workloads share one layer; a workload of another shape brings its own
    layer_wl = base if (wl.down, wl.d, wl.E, wl.f, wl.k) == (base.down, base.d, base.E, base.f, base.k) else wl
    W = synth.make_layer_weights(layer_wl, device="cuda")
    layer = ds4.Layer(layer_wl.d, layer_wl.E, layer_wl.f, layer_wl.k, max(4096, wl.T), W)
    del W
    torch.cuda.empty_cache()
    flush = L2Flush() if flushes_l2(wl) else None

    # ---- headline: device-resident inputs
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    res, acc, x, logits, out = measure_workload(ds4, layer, wl, args.steps, args.warmup, peaks, flush)
    barrier(ws)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_step = max_over_ranks(res["ms"], ws)
    value = job_value(ws, wl.T, ms_step)

    # ---- dominant kernel roofline
    roofline = dominant_roofline(res["kernels_ms"], acc, wl.name, peaks, fp8_peak, fp4_peak)

    # ---- end to end through the C ABI with host buffers
    xh = x.cpu().pin_memory()
    lh = logits.cpu().pin_memory()
    oh = torch.empty(wl.T, wl.d, dtype=torch.float32).pin_memory()
    for _ in range(max(1, args.warmup)):
        layer.forward_host(xh, lh, oh)
    e2e_ms = []
    for _ in range(args.steps):
        if flush:
            flush()
            torch.cuda.synchronize()
        t0 = time.perf_counter()
        layer.forward_host(xh, lh, oh)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_step = max_over_ranks(statistics.median(e2e_ms), ws)
    e2e = {"value": ws * wl.T / (e2e_step * 1e-3), "unit": "tokens/s",
           "h2d_bytes_per_step": int(xh.numel() * 2 + lh.numel() * 4),
           "d2h_bytes_per_step": int(oh.numel() * 4), "ms_per_step": e2e_step}

    # ---- the other workloads, same GPU (rank 0 reports them)
    also = {}
    if not args.no_extra:
        q2k_layer = None
        for name in ("decode1", "decode64", "prefill", "q2k", "q2k_decode1", "q2k_decode64"):
            if name == wl.name:
                continue
            other = synth.WORKLOADS[name]
            try:
                if other.down == "q2k" and layer_wl.down != "q2k":
                    if q2k_layer is None:  # one Q2_K layer (weight seed 4) serves its three workloads
                        qwl = synth.WORKLOADS["q2k"]
                        Wq = synth.make_layer_weights(qwl, device="cuda")
                        q2k_layer = ds4.Layer(qwl.d, qwl.E, qwl.f, qwl.k, qwl.T, Wq)
                        del Wq
                        torch.cuda.empty_cache()
                    lay2 = q2k_layer
                elif other.down != "q2k" and layer_wl.down == "q2k":
                    Wm = synth.make_layer_weights(other, device="cuda")
                    lay2 = ds4.Layer(other.d, other.E, other.f, other.k, max(4096, other.T), Wm)
                    del Wm
                    torch.cuda.empty_cache()
                else:
                    lay2 = layer
                fl = L2Flush() if flushes_l2(other) else None
                r, a, *_ = measure_workload(ds4, lay2, other, min(args.steps, 50), args.warmup, peaks, fl)
                if lay2 is not layer and lay2 is not q2k_layer:
                    lay2.close()
                    torch.cuda.empty_cache()
                also[name] = {k: v for k, v in r.items()}
                also[name]["algorithmic_bytes"] = a["total_bytes"]
                also[name]["roofline"] = dominant_roofline(r["kernels_ms"], a, name, peaks, fp8_peak, fp4_peak)
                if flushes_l2(other):
                    also[name]["l2"] = "flushed (512 MB write + read back) before every step"
            except Exception as exc:  # report, do not hide
                also[name] = {"error": str(exc)}
        if q2k_layer is not None:
            q2k_layer.close()
            torch.cuda.empty_cache()
        # the whole layer from x: router projection, routed experts, shared expert (fs = 2048, bf16)
        if layer_wl is base:
            try:
                Wx = {**synth.make_layer_weights(base, device="cuda"), **synth.make_dense_weights(base, 2048, device="cuda")}
                xl = ds4.Layer(base.d, base.E, base.f, base.k, 4096, Wx)
                del Wx
                torch.cuda.empty_cache()
                for name in ("decode1", "decode64", "prefill"):
                    other = synth.WORKLOADS[name]
                    fl = L2Flush() if flushes_l2(other) else None
                    r, a, *_ = measure_workload(ds4, xl, other, min(args.steps, 50), args.warmup, peaks, fl,
                                                with_x=True)
                    dense_bytes = (base.E * base.d + 3 * 2048 * base.d) * 2
                    r["algorithmic_bytes"] = a["total_bytes"] - other.T * base.E * 4 + dense_bytes
                    r["GBps"] = r["algorithmic_bytes"] / (r["ms"] * 1e-3) / 1e9
                    r["hbm_frac_of_measured"] = r["GBps"] / peaks["hbm_gbs"]
                    r["note"] = ("x in: router bf16 [256, 4096], routed MXFP4 experts, shared expert bf16 fs = 2048; "
                                 "bytes: routed weights touched + router + shared weights + x + out")
                    also[name + "_from_x"] = r
                xl.close()
                torch.cuda.empty_cache()
            except Exception as exc:
                also["from_x"] = {"error": str(exc)}

    # ---- CPU baseline: the oracle on a bounded sample (rank 0)
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(wl, layer_wl, budget_s=args.cpu_budget)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4(e2m1) x mxfp8(e4m3) -> fp32" if wl.T > 64 else "mxfp4(e2m1) x f16 -> fp32",
        "data": "synthetic (seeded; random-init MXFP4 weights, N(0,1) activations and logits)",
        "config": config_of(wl, ws),
        "achieved": {"algorithmic_bytes_per_step": acc["total_bytes"], "algorithmic_flops_per_step": acc["flops"],
                     "touched_experts": acc["U"], "GBps": res["GBps"], "TFLOPs": res["TFLOPs"],
                     "hbm_frac_of_measured": res["hbm_frac_of_measured"],
                     "tensor_frac_of_mxf8f6f4_peak": res["TFLOPs"] / fp8_peak,
                     "kernels_ms": res["kernels_ms"]},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": res["launches"] * args.steps,
        "clocks": clk,
        "workloads": also,
        "peaks": peaks,
    }
    if rank == 0:
        print(json.dumps(line))
    layer.close()
    if ws > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------- oracle
def oracle_tokens_per_s(wl: synth.Workload, W_host: dict, budget_s: float, seed_tokens=None):
    """Times the oracle on tokens of the workload until `budget_s` elapses."""
    import oracle
    inp = synth.make_inputs(wl, device="cpu")
    idx, w = oracle.route(inp["logits"].numpy(), wl.k)
    bits = inp["x"].view(torch.int16).numpy().view(np.uint16)
    act = oracle.ACT_EXACT if wl.T <= 64 else (oracle.ACT_MXFP8_X_ONLY if wl.down == "q2k" else oracle.ACT_MXFP8)
    dims = {"d": wl.d, "E": wl.E, "f": wl.f, "k": wl.k}
    rng = np.random.default_rng(0)
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        tok = int(rng.integers(0, wl.T))
        oracle.forward(dims, W_host, bits, idx, w, [tok], act)
        done += 1
    el = time.perf_counter() - t0
    return done / el, done, el, oracle.num_threads()


def oracle_weights(wl: synth.Workload) -> dict:
    # The oracle reads the same seeded bytes; generated on the GPU when there
    # is one (fast), else on the CPU.
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    W = synth.make_layer_weights(wl, device=dev)
    return {k: v.cpu().numpy() for k, v in W.items()}


def cpu_baseline(wl, layer_wl, budget_s: float) -> dict:
    Wh = oracle_weights(layer_wl)
    tps, n, el, cores = oracle_tokens_per_s(wl, Wh, budget_s)
    return {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} random tokens of the {wl.name} workload (each: its {wl.k} routed experts, "
                      f"full fp64 expert FFNs), {el:.1f} s of CPU time"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    base = synth.WORKLOADS["prefill"]
    layer_wl = base if (wl.down, wl.d, wl.E, wl.f, wl.k) == (base.down, base.d, base.E, base.f, base.k) else wl
    Wh = oracle_weights(layer_wl)
    per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_tokens_per_s(wl, Wh, per_step / 4)
    vals, toks, secs = [], 0, 0.0
    cores = 1
    for _ in range(args.steps):
        tps, n, el, cores = oracle_tokens_per_s(wl, Wh, per_step)
        vals.append(tps)
        toks += n
        secs += el
    value = toks / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        # a step is a bounded sample of the workload's tokens: this is the measured wall time of one
        "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": config_of(wl, ws),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{toks} random tokens of the {wl.name} workload over {args.steps} steps "
                                   f"({secs:.1f} s; each step a bounded sample, not the whole {wl.T}-token batch)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="prefill", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
