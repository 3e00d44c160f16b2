import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def ds4():
    """The compiled library (built in-tree if stale)."""
    import quantized_moe_expert_top_gb300 as m
    m.build()
    m.lib()
    return m


@pytest.fixture(scope="session")
def big_layer(ds4):
    """The full-size layer (d=4096, E=256, f=2048, k=8; weight seed 1) shared by
    the one-token decode, 64-token decode and 4096-token prefill workloads:
    device weights, a host copy for the oracle, and a library layer sized for
    4096 tokens."""
    import torch
    import synth
    wl = synth.WORKLOADS["prefill"]
    W = synth.make_layer_weights(wl, device="cuda")
    torch.cuda.synchronize()
    Wh = {k: v.cpu().numpy() for k, v in W.items()}
    layer = ds4.Layer(wl.d, wl.E, wl.f, wl.k, 4096, W)           # AUTO: DECODE_MMA for T <= 64, else PREFILL
    gemv = ds4.Layer(wl.d, wl.E, wl.f, wl.k, 64, W, force_path="decode")  # the CUDA-core GEMV decode path
    del W
    torch.cuda.empty_cache()
    yield {"wl": wl, "Wh": Wh, "layer": layer, "gemv": gemv}
    layer.close()
    gemv.close()
