"""The layer's original-precision parts on the GPU: the router projection
(logits = Wr . x) and the un-quantised shared expert added to every token's
output, against the oracle.  The routing decision is taken on fp32 logits on
both sides; tokens whose k-th and (k+1)-th logits are closer than the fp32
accumulation error could pick either expert and are left out (see
_sure_tokens)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_parity, bf16_bits, dims_of, host_weights

pytestmark = pytest.mark.gpu

TINY = synth.Workload("tiny_rs", 6, 256, 8, 128, 2, 31, 31, "normal")
MID = synth.Workload("mid_rs", 300, 512, 16, 384, 4, 32, 32, "normal")
# E = 6: the router block of the dense output is padded to 8 columns so that
# the shared expert's g and u columns stay 16-byte aligned
ODD_E = synth.Workload("odd_e_rs", 5, 256, 6, 128, 2, 33, 33, "normal")
ACT = {"decode": oracle.ACT_EXACT, "decode_mma": oracle.ACT_EXACT, "prefill": oracle.ACT_MXFP8}


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _sure_tokens(ref_logits32: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th logits are more than 1e-4 apart: two orders
    of magnitude above the fp32 accumulation error of the GPU's logits, so their
    selection is the oracle's on both sides.  A near-tie token may pick either
    expert (both are correct to fp32), so it is left out of the comparisons."""
    srt = -np.sort(-ref_logits32, axis=1)
    return (srt[:, k - 1] - srt[:, k]) > 1e-4


@pytest.mark.parametrize("path", ["decode", "decode_mma", "prefill"])
@pytest.mark.parametrize("wl,fs", [(TINY, 128), (MID, 384), (ODD_E, 64)], ids=["tiny", "mid", "odd_e"])
def test_router_and_shared_expert_from_x(ds4, wl, fs, path):
    W = synth.make_layer_weights(wl, device="cuda")
    D = synth.make_dense_weights(wl, fs, device="cuda")
    x = synth.make_x(wl, device="cuda")
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, wl.T, {**W, **D}, force_path=path)
    out = layer.forward_x(x)
    lg = layer.logits()
    r = layer.routing()
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    # logits: bf16 products summed in fp32 vs the exact sum
    ref_lg = oracle.router_logits(_bits(D["router"]), bf16_bits(x))
    assert np.abs(lg.cpu().numpy() - ref_lg).max() <= 1e-5 * (1 + np.abs(ref_lg).max())
    ref32 = ref_lg.astype(np.float32)
    sure = _sure_tokens(ref32, wl.k)
    assert sure.mean() >= 0.95
    idx, w = oracle.route(ref32, wl.k)
    assert np.array_equal(r["topk_idx"].cpu().numpy()[sure], idx[sure])
    # output: routed experts + the shared expert
    toks = [int(t) for t in np.nonzero(sure)[0]]
    ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(x), idx, w, toks, ACT[path])
    ref += oracle.shared_ffn(_bits(D["shared_gate"]), _bits(D["shared_up"]), _bits(D["shared_down"]), bf16_bits(x), toks)
    assert_parity(out.cpu().numpy()[toks], ref, f"{wl.name} {path}")
    layer.close()


def test_shared_expert_with_given_logits(ds4):
    """No router: ds4moe_forward routes on the given logits and still adds the
    shared expert; the x-only call is unsupported."""
    wl, fs = TINY, 64
    W = synth.make_layer_weights(wl, device="cuda")
    D = synth.make_dense_weights(wl, fs, device="cuda", router=False)
    inp = synth.make_inputs(wl, device="cuda")
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, wl.T, {**W, **D})
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    toks = list(range(wl.T))
    ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(inp["x"]), idx, w, toks, oracle.ACT_EXACT)
    ref += oracle.shared_ffn(_bits(D["shared_gate"]), _bits(D["shared_up"]), _bits(D["shared_down"]),
                             bf16_bits(inp["x"]), toks)
    assert_parity(out.cpu().numpy(), ref, "shared, given logits")
    names = [ds4.lib().ds4moe_kernel_name(layer._h, wl.T, i) for i in range(12)]
    names = [n for n in names if n is not None]
    assert names[:2] == [b"dense_in", b"shared_swiglu"] and names[-1] == b"shared_down"
    assert layer.launches_per_forward(wl.T) == len(names)
    with pytest.raises(ds4.Ds4moeError) as ei:
        layer.forward_x(inp["x"])
    assert ei.value.code == ds4.ERR_UNSUPPORTED
    layer.close()


@pytest.fixture(scope="module")
def full_layer(ds4):
    """The full-size layer (routed weights of seed 1) with a router and a shared
    expert of intermediate size 2048."""
    wl = synth.WORKLOADS["prefill"]
    W = synth.make_layer_weights(wl, device="cuda")
    D = synth.make_dense_weights(wl, 2048, device="cuda")
    torch.cuda.synchronize()
    Wh = host_weights(W)
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, 4096, {**W, **D})
    del W
    torch.cuda.empty_cache()
    yield wl, Wh, {k: _bits(v) for k, v in D.items()}, layer
    layer.close()


@pytest.mark.parametrize("name,ntok", [("decode1", None), ("decode64", None), ("prefill", 12)])
def test_full_size_router_and_shared_expert(ds4, full_layer, name, ntok):
    wl0, Wh, Db, layer = full_layer
    wl = synth.WORKLOADS[name]
    x = synth.make_x(wl, device="cuda")
    out = layer.forward_x(x)
    r = layer.routing()
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    ref_lg = oracle.router_logits(Db["router"], bf16_bits(x)).astype(np.float32)
    idx, w = oracle.route(ref_lg, wl.k)
    sure = _sure_tokens(ref_lg, wl.k)
    assert sure.mean() >= 0.95
    got_idx = r["topk_idx"].cpu().numpy()
    assert np.array_equal(got_idx[sure], idx[sure])
    toks = np.nonzero(sure)[0]
    if ntok is not None:
        toks = toks[np.linspace(0, toks.size - 1, ntok).astype(int)]
    toks = [int(t) for t in toks]
    act = oracle.ACT_MXFP8 if wl.T > 64 else oracle.ACT_EXACT
    ref = oracle.forward(dims_of(wl), Wh, bf16_bits(x), idx, w, toks, act)
    ref += oracle.shared_ffn(Db["shared_gate"], Db["shared_up"], Db["shared_down"], bf16_bits(x), toks)
    assert_parity(out.cpu().numpy()[toks], ref, name)
