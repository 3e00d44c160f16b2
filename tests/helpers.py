"""Shared test helpers: building layers from the seeded generator, running the
oracle on the same bytes, and the parity metrics."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Output tolerance of the layer (floating point): max |err| <= 2e-2 * rms(ref)
# and sum|err| / sum|ref| <= 5e-3; routing weights within 1e-6.
MAX_ERR_RMS = 2e-2
MEAN_REL = 5e-3
W_TOL = 1e-6


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host_weights(W: dict) -> dict:
    return {k: v.detach().cpu().numpy() for k, v in W.items()}


def dims_of(wl: synth.Workload) -> dict:
    return {"d": wl.d, "E": wl.E, "f": wl.f, "k": wl.k}


def parity_metrics(out_gpu: np.ndarray, ref: np.ndarray) -> dict:
    out_gpu = np.asarray(out_gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(out_gpu - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return {
        "max_err": float(err.max()),
        "rms_ref": rms,
        "max_err_over_rms": float(err.max() / rms) if rms > 0 else float("inf"),
        "mean_rel": float(err.sum() / np.abs(ref).sum()),
        "median_rel": float(np.median(err / np.maximum(np.abs(ref), 1e-30))),
        "finite": bool(np.isfinite(out_gpu).all()),
    }


def assert_parity(out_gpu, ref, what=""):
    m = parity_metrics(out_gpu, ref)
    assert m["finite"], (what, m)
    assert m["max_err_over_rms"] <= MAX_ERR_RMS, (what, m)
    assert m["mean_rel"] <= MEAN_REL, (what, m)
    return m


def sample_tokens(idx: np.ndarray, counts: np.ndarray, n: int, seed: int = 0) -> list:
    """Tokens for sampled parity: first, last, some routed to the most and the
    least loaded experts, and a seeded random remainder."""
    T = idx.shape[0]
    rng = np.random.default_rng(seed)
    pick = {0, T - 1}
    order = np.argsort(counts)
    for e in list(order[-2:]) + [x for x in order if counts[x] > 0][:2]:
        hits = np.nonzero((idx == e).any(axis=1))[0]
        if hits.size:
            pick.add(int(hits[0]))
            pick.add(int(hits[-1]))
    while len(pick) < min(n, T):
        pick.add(int(rng.integers(0, T)))
    return sorted(pick)
