"""The largest layer dimensions the library accepts, d_model = d_ff = 8192,
on every path against the oracle: the CUDA-core GEMV (its down ring then holds
one stage), the few-token GEMMs (T = 3 takes the single-block routing whose
shared-memory copy of the MXFP8 rows is at its maximum; T = 12 the routing
kernels), the prefill GEMMs, and the Q2_K down projection (32 super-blocks per
row).  Three or four experts keep the weights at about 300-400 MB."""
import pytest

import oracle
import synth
from helpers import assert_parity, bf16_bits, dims_of, host_weights

pytestmark = pytest.mark.gpu

MAX4 = synth.Workload("max_dims", 12, 8192, 4, 8192, 2, 51, 51, "normal")
MAX_Q2K = synth.Workload("max_dims_q2k", 12, 8192, 3, 8192, 2, 52, 52, "normal", "q2k")

ACT = {("mxfp4", "decode"): oracle.ACT_EXACT, ("mxfp4", "decode_mma"): oracle.ACT_EXACT,
       ("mxfp4", "prefill"): oracle.ACT_MXFP8, ("q2k", "decode_mma"): oracle.ACT_EXACT,
       ("q2k", "prefill"): oracle.ACT_MXFP8_X_ONLY}

CASES = [(MAX4, "decode", 12), (MAX4, "decode_mma", 3), (MAX4, "decode_mma", 12), (MAX4, "prefill", 12),
         (MAX_Q2K, "decode_mma", 12), (MAX_Q2K, "prefill", 12)]


@pytest.mark.parametrize("wl,path,T", CASES, ids=[f"{w.name}-{p}-T{t}" for w, p, t in CASES])
def test_max_dims(ds4, wl, path, T):
    W = synth.make_layer_weights(wl, device="cuda")
    inp = synth.make_inputs(wl, device="cuda", T=T)
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, wl.T, W, force_path=path)
    out = layer.forward(inp["x"], inp["logits"])
    assert layer.status() == ds4.OK
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    assert (layer.routing()["topk_idx"].cpu().numpy() == idx).all(), "expert selection"
    ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(inp["x"]), idx, w, list(range(T)),
                         ACT[(wl.down, path)])
    assert_parity(out.cpu().numpy(), ref, f"{wl.name} {path} T={T}")
    layer.close()
