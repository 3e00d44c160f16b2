"""Asymmetric 2-bit variant: MXFP4 gate/up with a Q2_K-style down projection
(dequantised to fp16 inside the down GEMM's operand load) vs the oracle, on
both tensor-core paths (few-token DECODE_MMA and PREFILL)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_parity, bf16_bits, coverage_tokens, dims_of, host_weights

pytestmark = pytest.mark.gpu

TINY_Q2K = synth.Workload("tinyq2k", 6, 256, 6, 256, 2, 12, 12, "perm", "q2k")
MID_Q2K = synth.Workload("midq2k", 500, 512, 8, 512, 2, 13, 13, "zipf", "q2k")  # chunks past 192 tokens


@pytest.mark.parametrize("path", ["prefill", "decode_mma"])
@pytest.mark.parametrize("wl", [TINY_Q2K, MID_Q2K], ids=lambda w: w.name)
def test_q2k_full_parity(ds4, wl, path):
    """Both tensor-core paths of a Q2_K layer: PREFILL (MXFP8 x, fp16 h) against
    the oracle's x-only MXFP8 mode, DECODE_MMA (split x, fp16 h) against its
    exact-activation mode."""
    W = synth.make_layer_weights(wl, device="cuda")
    inp = synth.make_inputs(wl, device="cuda")
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, wl.T, W, force_path=path)
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    act = oracle.ACT_MXFP8_X_ONLY if path == "prefill" else oracle.ACT_EXACT
    ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(inp["x"]), idx, w, list(range(wl.T)), act)
    assert_parity(out.cpu().numpy(), ref, f"{wl.name} {path}")
    layer.close()


def test_q2k_auto_path_choice(ds4):
    W = synth.make_layer_weights(TINY_Q2K, device="cuda")
    layer = ds4.Layer(TINY_Q2K.d, TINY_Q2K.E, TINY_Q2K.f, TINY_Q2K.k, 6, W, decode_max_tokens=4)
    assert layer.path_for(4) == ds4.PATH_DECODE_MMA and layer.path_for(5) == ds4.PATH_PREFILL
    names = [ds4.lib().ds4moe_kernel_name(layer._h, 1, i) for i in range(4)]
    assert names == [b"route_small", b"decode_mma_gateup", b"gemm_down", None]
    layer.close()


def test_q2k_gemv_path_is_rejected(ds4):
    W = synth.make_layer_weights(TINY_Q2K, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.Layer(TINY_Q2K.d, TINY_Q2K.E, TINY_Q2K.f, TINY_Q2K.k, 6, W, force_path="decode")
    assert ei.value.code == ds4.ERR_UNSUPPORTED


@pytest.fixture(scope="module")
def q2k_layer(ds4):
    """The full-size Q2_K layer (weight seed 4) for 1, 64 and 2048 tokens."""
    wl = synth.WORKLOADS["q2k"]
    W = synth.make_layer_weights(wl, device="cuda")
    torch.cuda.synchronize()
    Wh = host_weights(W)
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, wl.T, W)
    del W
    torch.cuda.empty_cache()
    yield wl, Wh, layer
    layer.close()


@pytest.mark.parametrize("name", ["q2k_decode1", "q2k_decode64"])
def test_q2k_decode_full_size_every_token(ds4, q2k_layer, name):
    wl0, Wh, layer = q2k_layer
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, device="cuda")
    assert layer.path_for(wl.T) == ds4.PATH_DECODE_MMA
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    ref = oracle.forward(dims_of(wl), Wh, bf16_bits(inp["x"]), idx, w, list(range(wl.T)), oracle.ACT_EXACT)
    assert_parity(out.cpu().numpy(), ref, name)


def test_q2k_2048_tokens_every_expert_and_chunk_end(ds4, q2k_layer):
    wl, Wh, layer = q2k_layer
    inp = synth.make_inputs(wl, device="cuda")
    assert layer.path_for(wl.T) == ds4.PATH_PREFILL
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
