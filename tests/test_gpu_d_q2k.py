"""Asymmetric 2-bit variant: MXFP4 gate/up with a Q2_K-style down projection
(dequantised to fp16 inside the down GEMM's operand load) vs the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_parity, bf16_bits, coverage_tokens, dims_of, host_weights

pytestmark = pytest.mark.gpu

TINY_Q2K = synth.Workload("tinyq2k", 6, 256, 6, 256, 2, 12, 12, "perm", "q2k")
MID_Q2K = synth.Workload("midq2k", 500, 512, 8, 512, 2, 13, 13, "zipf", "q2k")  # chunks past 192 tokens


@pytest.mark.parametrize("wl", [TINY_Q2K, MID_Q2K], ids=lambda w: w.name)
def test_q2k_full_parity(ds4, wl):
    W = synth.make_layer_weights(wl, device="cuda")
    inp = synth.make_inputs(wl, device="cuda")
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, wl.T, W)
    assert layer.path_for(1) == ds4.PATH_PREFILL  # a Q2_K layer always takes the GEMM path
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(inp["x"]), idx, w, list(range(wl.T)),
                         oracle.ACT_MXFP8_X_ONLY)
    assert_parity(out.cpu().numpy(), ref, wl.name)
    layer.close()


@pytest.mark.parametrize("path", ["decode", "decode_mma"])
def test_q2k_decode_paths_are_rejected(ds4, path):
    W = synth.make_layer_weights(TINY_Q2K, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.Layer(TINY_Q2K.d, TINY_Q2K.E, TINY_Q2K.f, TINY_Q2K.k, 6, W, force_path=path)
    assert ei.value.code == ds4.ERR_UNSUPPORTED


def test_q2k_2048_tokens_every_expert_and_chunk_end(ds4):
    wl = synth.WORKLOADS["q2k"]
    W = synth.make_layer_weights(wl, device="cuda")
    torch.cuda.synchronize()
    Wh = host_weights(W)
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, wl.T, W)
    del W
    torch.cuda.empty_cache()
    inp = synth.make_inputs(wl, device="cuda")
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    out = out.cpu().numpy()
    assert np.isfinite(out).all()
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    toks = coverage_tokens(idx, wl.E)  # every expert, both ends of its 128-token chunks (~170 tokens)
    assert set(idx[toks].ravel().tolist()) == set(range(wl.E))
    ref = oracle.forward(dims_of(wl), Wh, bf16_bits(inp["x"]), idx, w, toks, oracle.ACT_MXFP8_X_ONLY)
    assert_parity(out[toks], ref, "q2k")
    layer.close()
