"""Edge cases of the C ABI on the GPU: empty calls, size limits, alignment,
host-buffer calls, launch counts."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_parity, bf16_bits, dims_of, host_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny(ds4):
    wl = synth.WORKLOADS["tiny"]
    W = synth.make_layer_weights(wl, device="cuda")
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, 16, W, decode_max_tokens=4)
    yield wl, W, layer
    layer.close()


def test_empty_call_is_a_no_op(ds4, tiny):
    wl, _, layer = tiny
    x = torch.empty(0, wl.d, dtype=torch.bfloat16, device="cuda")
    lg = torch.empty(0, wl.E, dtype=torch.float32, device="cuda")
    out = layer.forward(x, lg)
    assert out.shape == (0, wl.d)
    assert layer.launches_per_forward(0) == 0
    assert layer.status() == ds4.OK


def test_too_many_tokens_rejected(ds4, tiny):
    wl, _, layer = tiny
    x = torch.zeros(17, wl.d, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(17, wl.E, dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        layer.forward(x, lg)
    assert ei.value.code == ds4.ERR_TOO_MANY_TOKENS


def test_misaligned_pointer_rejected(ds4, tiny):
    wl, _, layer = tiny
    buf = torch.zeros(4 * wl.d + 8, dtype=torch.bfloat16, device="cuda")
    x = buf[1:1 + 4 * wl.d].view(4, wl.d)  # 2-byte offset
    lg = torch.zeros(4, wl.E, dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        layer.forward(x, lg)
    assert ei.value.code == ds4.ERR_INVALID_ARG


def test_out_overlapping_an_input_is_rejected(ds4, tiny):
    wl, _, layer = tiny
    buf = torch.zeros(4 * wl.d * 4 + 4 * wl.E * 4, dtype=torch.uint8, device="cuda")
    out = buf[:4 * wl.d * 4].view(torch.float32).view(4, wl.d)
    x = buf[:4 * wl.d * 2].view(torch.bfloat16).view(4, wl.d)            # x inside out
    lg = torch.zeros(4, wl.E, dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        layer.forward(x, lg, out)
    assert ei.value.code == ds4.ERR_INVALID_ARG
    x2 = torch.zeros(4, wl.d, dtype=torch.bfloat16, device="cuda")
    lg2 = buf[4 * wl.d * 4 - 64:4 * wl.d * 4 - 64 + 4 * wl.E * 4].view(torch.float32).view(4, wl.E)  # logits overlap out's tail
    with pytest.raises(ds4.Ds4moeError) as ei:
        layer.forward(x2, lg2, out)
    assert ei.value.code == ds4.ERR_INVALID_ARG


def test_path_choice_and_launch_counts(ds4, tiny):
    _, _, layer = tiny
    assert layer.path_for(4) == ds4.PATH_DECODE_MMA
    assert layer.path_for(5) == ds4.PATH_PREFILL
    assert layer.path_for(17) == ds4.ERR_TOO_MANY_TOKENS
    # up to 4 tokens, routing and the activation quantisation are one launch
    assert layer.launches_per_forward(4) == 3
    assert layer.launches_per_forward(16) == 5
    names = [ds4.lib().ds4moe_kernel_name(layer._h, 4, i) for i in range(4)]
    assert names == [b"route_small", b"decode_mma_gateup", b"decode_mma_down", None]
    names = [ds4.lib().ds4moe_kernel_name(layer._h, 16, i) for i in range(6)]
    assert names == [b"route_topk", b"route_group", b"act_quant", b"gemm_gateup", b"gemm_down", None]


@pytest.mark.parametrize("T", [4, 16])
def test_host_call_matches_device_call(ds4, tiny, T):
    wl, W, layer = tiny
    inp = synth.make_inputs(wl, device="cpu", T=T)
    out_h = layer.forward_host(inp["x"].pin_memory(), inp["logits"].pin_memory())
    out_d = layer.forward(inp["x"].cuda(), inp["logits"].cuda()).cpu()
    assert torch.allclose(out_h, out_d, rtol=1e-5, atol=1e-6)
    act = oracle.ACT_EXACT if T <= 4 else oracle.ACT_MXFP8  # T <= 4: DECODE_MMA (exact-activation mode)
    idx, w = oracle.route(inp["logits"].numpy(), wl.k)
    ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(inp["x"]), idx, w, list(range(T)), act)
    assert_parity(out_h.numpy(), ref, f"host T={T}")


def test_layer_at_max_tokens_both_paths(ds4):
    wl = synth.Workload("maxT", 33, 256, 16, 256, 4, 9, 9, "normal")
    W = synth.make_layer_weights(wl, device="cuda")
    inp = synth.make_inputs(wl, device="cuda")
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    for path, act in (("decode", oracle.ACT_EXACT), ("decode_mma", oracle.ACT_EXACT), ("prefill", oracle.ACT_MXFP8)):
        layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, 33, W, force_path=path)
        out = layer.forward(inp["x"], inp["logits"])
        torch.cuda.synchronize()
        assert layer.status() == ds4.OK
        ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(inp["x"]), idx, w, list(range(33)), act)
        assert_parity(out.cpu().numpy(), ref, path)
        layer.close()
