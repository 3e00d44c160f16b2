"""Routing on the GPU vs the oracle: selected experts, the grouping offsets and
the (expert, token) permutation must match bit for bit; weights within 1e-6."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _routing_layer(ds4, wl, T, path):
    # Routing does not depend on d or f: a small layer with the workload's E and k.
    small = synth.Workload("r", T, 128, wl.E, 128, wl.k, wl.seed, 7, wl.routing)
    W = synth.make_layer_weights(small, device="cuda")
    return ds4.Layer(128, wl.E, 128, wl.k, T, W, force_path=path)


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode64", "prefill", "q2k"])
@pytest.mark.parametrize("path", ["decode", "decode_mma", "prefill"])
def test_routing_matches_oracle(ds4, name, path):
    wl = synth.WORKLOADS[name]
    logits = synth.make_logits(wl, device="cuda")
    T = logits.shape[0]
    x = torch.randn(T, 128, device="cuda").to(torch.bfloat16)
    layer = _routing_layer(ds4, wl, T, path)
    layer.forward(x, logits)
    r = layer.routing()
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    idx_ref, w_ref = oracle.route(logits.cpu().numpy(), wl.k)
    G = oracle.group(idx_ref, wl.E)
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx_ref)
    assert np.array_equal(r["offsets"].cpu().numpy(), G["offsets"])
    assert np.array_equal(r["perm_tok"].cpu().numpy(), G["perm_tok"])
    w = r["topk_w"].cpu().numpy().astype(np.float64)
    assert np.abs(w - w_ref).max() <= 1e-6
    assert np.abs(w.sum(1) - 1.0).max() <= 1e-6
    # every token appears exactly k times in the permutation
    assert np.array_equal(np.bincount(r["perm_tok"].cpu().numpy(), minlength=T), np.full(T, wl.k))
    layer.close()


def test_routing_ties_and_nan_rank_like_oracle(ds4):
    E, k, T = 64, 6, 40
    g = torch.Generator().manual_seed(3)
    logits = torch.randint(-3, 4, (T, E), generator=g).to(torch.float32)  # many exact ties
    logits[5, :] = 1.0          # all equal: lowest indices win
    logits[6, 10] = float("nan")  # NaN ranks like -inf
    logits[7, :] = -0.0
    logits[7, 3] = 0.0
    wl = synth.Workload("ties", T, 128, E, 128, k, 0, 0, "normal")
    layer = _routing_layer(ds4, wl, T, "decode")
    x = torch.randn(T, 128, device="cuda").to(torch.bfloat16)
    layer.forward(x, logits.cuda())
    r = layer.routing()
    idx_ref, w_ref = oracle.route(logits.numpy(), k)
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx_ref)
    assert list(idx_ref[5]) == list(range(k))
    G = oracle.group(idx_ref, E)
    assert np.array_equal(r["perm_tok"].cpu().numpy(), G["perm_tok"])
    layer.close()
