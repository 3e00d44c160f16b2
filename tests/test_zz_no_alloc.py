"""ds4moe_route_noalloc: routing for callers that cannot allocate device
memory at routing time (a memory plan fixed at start-up, or a serving loop
that cannot afford cudaMalloc's implicit synchronisation).  It must give the
same routing as the layer's forward call, on repeated calls that share its one
file-scope scratch array, and reject sizes beyond that array."""
import numpy as np
import pytest
import torch

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
def test_noalloc_routing_matches_forward_routing_twice(ds4, name):
    wl = synth.WORKLOADS[name]  # q2k: 2048 tokens x top-8 = the array's 16384-pair limit
    logits = synth.make_logits(wl, device="cuda")
    ref = _layer_routing(ds4, wl, logits)
    other = synth.make_logits(synth.WORKLOADS["decode1"], device="cuda")[:, :wl.E].contiguous()
    for call in range(2):
        got = ds4.route_noalloc(logits, wl.k)
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in got.items()}
        assert np.array_equal(got["topk_idx"], ref["topk_idx"]), call
        assert np.abs(got["topk_w"] - ref["topk_w"]).max() <= 1e-6, call
        assert np.array_equal(got["offsets"], ref["offsets"]), call
        assert np.array_equal(got["perm_tok"], ref["perm_tok"]), call
        ds4.route_noalloc(other, min(wl.k, other.shape[1]))  # leave different contents in the scratch


def test_noalloc_rejects_sizes_beyond_its_array(ds4):
    logits = torch.zeros(2049, 256, dtype=torch.float32, device="cuda")
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.route_noalloc(logits, 8)
    assert ei.value.code == ds4.ERR_TOO_MANY_TOKENS
    with pytest.raises(ds4.Ds4moeError) as ei:
        ds4.route_noalloc(torch.zeros(4, 300, device="cuda"), 2)
    assert ei.value.code == ds4.ERR_INVALID_ARG
