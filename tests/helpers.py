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


def coverage_tokens(idx: np.ndarray, E: int, chunk: int = 128) -> list:
    """Tokens for sampled parity at full size that reach every expert and both
    ends of every block of `chunk` consecutive tokens of an expert (the grouped
    GEMMs split an expert's token columns into chunks that start on 128-token
    boundaries): for each expert with n routed tokens in (expert, token) order,
    the tokens at positions 0 and n - 1 and at b - 1 and b for every multiple b
    of `chunk` below n."""
    pick = set()
    for e in range(E):
        toks = np.nonzero((idx == e).any(axis=1))[0]
        n = toks.size
        if n == 0:
            continue
        pos = {0, n - 1}
        for b in range(chunk, n, chunk):
            pos.update((b - 1, b))
        pick.update(int(toks[p]) for p in pos)
    return sorted(pick)
