"""Degenerate routing shapes on every path, against the oracle: k = E (every
token selects every expert, so each expert's tokens are the whole batch) and
k = 1 with several experts (a plain argmax route, softmax weight 1), for the
MXFP4 layer (GEMV, DECODE_MMA, PREFILL) and the Q2_K layer (DECODE_MMA,
PREFILL); and a one-token, one-expert call (the smallest GEMM: one 16-row
token tile of which one row is used)."""
import pytest
import torch

import oracle
import synth
from helpers import assert_parity, bf16_bits, dims_of, host_weights

pytestmark = pytest.mark.gpu

ALL_E = synth.Workload("all_e", 37, 256, 4, 256, 4, 41, 41, "normal")           # k = E = 4
TOP1 = synth.Workload("top1", 90, 256, 8, 128, 1, 42, 42, "normal")             # k = 1 of 8
ONE = synth.Workload("one", 1, 256, 1, 128, 1, 43, 43, "normal")                # T = 1, E = k = 1
ALL_E_Q2K = synth.Workload("all_e_q2k", 21, 256, 4, 256, 4, 44, 44, "normal", "q2k")
TOP1_Q2K = synth.Workload("top1_q2k", 70, 256, 6, 256, 1, 45, 45, "normal", "q2k")

ACT = {("mxfp4", "decode"): oracle.ACT_EXACT, ("mxfp4", "decode_mma"): oracle.ACT_EXACT,
       ("mxfp4", "prefill"): oracle.ACT_MXFP8, ("q2k", "decode_mma"): oracle.ACT_EXACT,
       ("q2k", "prefill"): oracle.ACT_MXFP8_X_ONLY}

CASES = [(wl, path) for wl in (ALL_E, TOP1, ONE) for path in ("decode", "decode_mma", "prefill")] + \
        [(wl, path) for wl in (ALL_E_Q2K, TOP1_Q2K) for path in ("decode_mma", "prefill")]


@pytest.mark.parametrize("wl,path", CASES, ids=[f"{w.name}-{p}" for w, p in CASES])
def test_degenerate_routing_shapes(ds4, wl, path):
    W = synth.make_layer_weights(wl, device="cuda")
    inp = synth.make_inputs(wl, device="cuda")
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, max(wl.T, 1), W, force_path=path)
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    routing = layer.routing()
    assert (routing["topk_idx"].cpu().numpy() == idx).all(), "expert selection"
    if wl.k == wl.E:
        assert (routing["offsets"].cpu().numpy() == [t * wl.T for t in range(wl.E + 1)]).all()
    ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(inp["x"]), idx, w, list(range(wl.T)),
                         ACT[(wl.down, path)])
    assert_parity(out.cpu().numpy(), ref, f"{wl.name} {path}")
    layer.close()
