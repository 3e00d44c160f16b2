"""Prefill (grouped tcgen05 GEMM) path vs the oracle in its MXFP8 mode."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_parity, bf16_bits, coverage_tokens, dims_of, host_weights
from test_gpu_b_decode import MID, UNIT, _run

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", [synth.WORKLOADS["tiny"], MID, UNIT], ids=lambda w: w.name)
def test_prefill_path_full_parity(ds4, wl):
    out, ref = _run(ds4, wl, "prefill")
    assert_parity(out, ref, wl.name)


def test_prefill_chunks_past_256_tokens(ds4):
    # one expert receives > 256 tokens: gate/up and down both split its columns
    wl = synth.Workload("hot", 600, 256, 4, 256, 1, 8, 8, "zipf")
    out, ref = _run(ds4, wl, "prefill")
    idx, _ = oracle.route(synth.make_logits(wl).numpy(), 1)
    assert_parity(out, ref, "hot")


def test_prefill_4096_tokens_every_expert_and_chunk_end(ds4, big_layer):
    wl = synth.WORKLOADS["prefill"]
    layer = big_layer["layer"]
    inp = synth.make_inputs(wl, device="cuda")
    assert layer.path_for(4096) == ds4.PATH_PREFILL
    out = layer.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert layer.status() == ds4.OK
    out = out.cpu().numpy()
    assert np.isfinite(out).all()
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    toks = coverage_tokens(idx, wl.E)  # every expert, both ends of its 128-token chunks (~340 tokens)
    assert set(idx[toks].ravel().tolist()) == set(range(wl.E))
    ref = oracle.forward(dims_of(wl), big_layer["Wh"], bf16_bits(inp["x"]), idx, w, toks, oracle.ACT_MXFP8)
    assert_parity(out[toks], ref, "prefill")
