"""ds4moe_route_noalloc: routing for callers that cannot allocate device
memory at routing time (a memory plan fixed at start-up, or a serving loop
that cannot afford cudaMalloc's implicit synchronisation).  Its results must
equal the oracle's routing and grouping and the layer's own routing, on
repeated calls that share its one file-scope scratch array, and it must reject
sizes beyond that array."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _layer_routing(ds4, wl, logits):
    small = synth.Workload("r", logits.shape[0], 128, wl.E, 128, wl.k, wl.seed, 7, wl.routing)
    W = synth.make_layer_weights(small, device="cuda")
    layer = ds4.Layer(128, wl.E, 128, wl.k, logits.shape[0], W, force_path="decode")
    x = torch.zeros(logits.shape[0], 128, dtype=torch.bfloat16, device="cuda")
    layer.forward(x, logits)
    r = layer.routing()
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    layer.close()
    return {k: v.cpu().numpy() for k, v in r.items()}


@pytest.mark.parametrize("name", ["tiny", "decode64", "q2k"])
def test_noalloc_routing_matches_oracle_and_forward_twice(ds4, name):
    wl = synth.WORKLOADS[name]  # q2k: 2048 tokens x top-8 = the array's 16384-pair limit
    logits = synth.make_logits(wl, device="cuda")
    idx_ref, w_ref = oracle.route(logits.cpu().numpy(), wl.k)
    G = oracle.group(idx_ref, wl.E)
    layer_r = _layer_routing(ds4, wl, logits)
    other = synth.make_logits(synth.WORKLOADS["decode1"], device="cuda")[:, :wl.E].contiguous()
    for call in range(2):
        got = ds4.route_noalloc(logits, wl.k)
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in got.items()}
        assert np.array_equal(got["topk_idx"], idx_ref), call
        assert np.abs(got["topk_w"].astype(np.float64) - w_ref).max() <= 1e-6, call
        assert np.array_equal(got["offsets"], G["offsets"]), call
        assert np.array_equal(got["perm_tok"], G["perm_tok"]), call
        for key in ("topk_idx", "offsets", "perm_tok"):
            assert np.array_equal(got[key], layer_r[key]), (call, key)
        ds4.route_noalloc(other, min(wl.k, other.shape[1]))  # leave different contents in the scratch


def test_noalloc_empty_call_zeroes_offsets(ds4):
    offs = ds4.route_noalloc(torch.zeros(0, 16, dtype=torch.float32, device="cuda"), 4)["offsets"]
    torch.cuda.synchronize()
    assert offs.shape == (17,) and not offs.any()


def test_noalloc_rejects_sizes_beyond_its_array(ds4):
    logits = torch.zeros(2049, 256, dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.route_noalloc(logits, 8)
    assert ei.value.code == ds4.ERR_TOO_MANY_TOKENS
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.route_noalloc(torch.zeros(4, 300, device="cuda"), 2)
    assert ei.value.code == ds4.ERR_INVALID_ARG
