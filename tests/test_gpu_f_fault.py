"""Failure detection without a GPU fault: a test-only knob makes the first
CTA pair of the gate/up GEMM wait on a barrier that nothing arrives on, so its
bounded waits run out (~1 ms).  The kernel records the timeout in the layer's
status word, lets every copy it issued land and exits cleanly; the host reads
DS4MOE_ERR_DEVICE_TIMEOUT and the GPU stays usable."""
import pytest
import torch

import oracle
import synth
from helpers import assert_parity, bf16_bits, dims_of, host_weights

pytestmark = pytest.mark.gpu


def test_unarrived_barrier_times_out_and_reports(ds4):
    wl = synth.WORKLOADS["tiny"]
    W = synth.make_layer_weights(wl, device="cuda")
    inp = synth.make_inputs(wl, device="cuda")
    bad = ds4.Layer(wl.d, wl.E, wl.f, wl.k, wl.T, W, force_path="prefill", debug_fault=1)
    bad.forward(inp["x"], inp["logits"])
    assert bad.status() == ds4.ERR_DEVICE_TIMEOUT
    assert bad.status() == ds4.OK  # the status word was cleared by the read
    bad.close()
    # the context and the GPU are still usable
    good = ds4.Layer(wl.d, wl.E, wl.f, wl.k, wl.T, W, force_path="prefill")
    out = good.forward(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert good.status() == ds4.OK
    idx, w = oracle.route(inp["logits"].cpu().numpy(), wl.k)
    ref = oracle.forward(dims_of(wl), host_weights(W), bf16_bits(inp["x"]), idx, w, list(range(wl.T)),
                         oracle.ACT_MXFP8)
    assert_parity(out.cpu().numpy(), ref, "after fault")
    good.close()
