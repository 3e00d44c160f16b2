"""Few-token decode paths vs the oracle in its exact-activation mode: the
CUDA-core GEMV path (forced) and the split-precision tensor-core path
(DECODE_MMA, the default for T <= 64)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_parity, bf16_bits, dims_of, host_weights

pytestmark = pytest.mark.gpu

MID = synth.Workload("mid", 700, 512, 8, 384, 2, 5, 5, "zipf")     # several tiles, ragged, skewed
UNIT = synth.Workload("unit", 5, 256, 1, 256, 1, 6, 6, "normal")   # E = 1, k = 1: dense SwiGLU FFN


def _run(ds4, wl, path, T=None):
    W = synth.make_layer_weights(wl, device="cuda")
    inp = synth.make_inputs(wl, device="cuda", T=T)
    T = inp["x"].shape[0]
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, T, W, force_path=path)
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    act = oracle.ACT_MXFP8 if path == "prefill" else oracle.ACT_EXACT
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(inp["x"]), idx, w, list(range(T)), act)
    layer.close()
    return out.cpu().numpy(), ref


@pytest.mark.parametrize("path", ["decode", "decode_mma"])
@pytest.mark.parametrize("wl", [synth.WORKLOADS["tiny"], MID, UNIT], ids=lambda w: w.name)
def test_decode_paths_full_parity(ds4, wl, path):
    out, ref = _run(ds4, wl, path)
    assert_parity(out, ref, f"{wl.name} {path}")


@pytest.mark.parametrize("which", ["layer", "gemv"])
def test_decode_one_token_full_size(ds4, big_layer, which):
    wl = synth.WORKLOADS["decode1"]
    layer = big_layer[which]
    inp = synth.make_inputs(wl, device="cuda")
    assert layer.path_for(1) == (ds4.PATH_DECODE_MMA if which == "layer" else ds4.PATH_DECODE)
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    ref = oracle.forward(dims_of(wl), big_layer["Wh"], bf16_bits(inp["x"]), idx, w, [0], oracle.ACT_EXACT)
    assert_parity(out.cpu().numpy(), ref, "decode1")


@pytest.mark.parametrize("which", ["layer", "gemv"])
def test_decode_64_tokens_zipf_full_size(ds4, big_layer, which):
    wl = synth.WORKLOADS["decode64"]
    layer = big_layer[which]
    inp = synth.make_inputs(wl, device="cuda")
    assert layer.path_for(64) == (ds4.PATH_DECODE_MMA if which == "layer" else ds4.PATH_DECODE)
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    assert counts.max() > 16  # the Zipf prior concentrates load
    ref = oracle.forward(dims_of(wl), big_layer["Wh"], bf16_bits(inp["x"]), idx, w, list(range(64)),
                         oracle.ACT_EXACT)
    assert_parity(out.cpu().numpy(), ref, "decode64")
