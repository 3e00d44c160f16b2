"""CPU checks of the C ABI: the library loads, exports every function that
include/ds4moe.h declares, and rejects bad arguments on the host before any
device work.  No compute calls are made."""
import ctypes

import quantized_moe_expert_top_gb300 as m


def test_library_builds_and_exports_every_header_symbol(ds4):
    names = m.header_functions()
    assert len(names) >= 10
    L = ds4.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings(ds4):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = ds4.status_string(code)
        assert s and s != "unknown status"
    assert ds4.status_string(-99) == "unknown status"


def test_defaults(ds4):
    c = ds4.default_config()
    assert (c.d_model, c.n_experts, c.d_ff, c.top_k, c.max_tokens) == (0, 0, 0, 0, 0)
    assert c.decode_max_tokens == 64 and c.wait_timeout_ms == 2000
    assert c.force_path == ds4.PATH_AUTO and c.debug_fault == 0


def test_null_handles(ds4):
    L = ds4.lib()
    assert L.ds4moe_path_for(None, 1) == ds4.ERR_INVALID_ARG
    assert L.ds4moe_launches_per_forward(None, 1) == ds4.ERR_INVALID_ARG
    assert L.ds4moe_forward(None, None, None, None, 1, None) == ds4.ERR_INVALID_ARG
    assert L.ds4moe_get_status(None) == ds4.ERR_INVALID_ARG
    assert L.ds4moe_get_routing(None, None, None, None, None, None) == ds4.ERR_INVALID_ARG
    L.ds4moe_destroy(None)  # NULL-safe


def _create(ds4, **kw):
    c = ds4.default_config()
    c.d_model, c.n_experts, c.d_ff, c.top_k, c.max_tokens = 256, 8, 128, 2, 4
    for k, v in kw.items():
        setattr(c, k, v)
    w = ds4.WeightPtrs()
    buf = (ctypes.c_uint8 * 64)()
    for n in ("gate_codes", "gate_scales", "up_codes", "up_scales", "down_codes", "down_scales"):
        setattr(w, n, ctypes.addressof(buf))
    h = ctypes.c_void_p(123)
    rc = ds4.lib().ds4moe_layer_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h))
    return rc, h


def test_create_rejects_bad_shapes_on_host(ds4):
    cases = [
        ({"d_model": 100}, ds4.ERR_UNSUPPORTED),      # not a multiple of 128
        ({"d_ff": 64}, ds4.ERR_UNSUPPORTED),
        ({"n_experts": 0}, ds4.ERR_UNSUPPORTED),
        ({"n_experts": 300}, ds4.ERR_UNSUPPORTED),
        ({"top_k": 9}, ds4.ERR_UNSUPPORTED),
        ({"top_k": 0}, ds4.ERR_UNSUPPORTED),
        ({"max_tokens": 0}, ds4.ERR_INVALID_ARG),
        ({"down_format": 7}, ds4.ERR_INVALID_ARG),
        ({"down_format": 1, "d_ff": 384}, ds4.ERR_UNSUPPORTED),  # Q2_K needs f % 256 == 0
        ({"force_path": 5}, ds4.ERR_INVALID_ARG),
        ({"wait_timeout_ms": 0}, ds4.ERR_INVALID_ARG),
        ({"decode_max_tokens": -1}, ds4.ERR_INVALID_ARG),
    ]
    for kw, want in cases:
        rc, h = _create(ds4, **kw)
        assert rc == want, (kw, rc)
        assert h.value is None, kw  # *out cleared on failure


def test_create_rejects_null_weights(ds4):
    c = ds4.default_config()
    c.d_model, c.n_experts, c.d_ff, c.top_k, c.max_tokens = 256, 8, 128, 2, 4
    w = ds4.WeightPtrs()
    h = ctypes.c_void_p()
    assert ds4.lib().ds4moe_layer_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)) == ds4.ERR_INVALID_ARG
    assert ds4.lib().ds4moe_layer_create(ctypes.byref(c), None, ctypes.byref(h)) == ds4.ERR_INVALID_ARG
    assert ds4.lib().ds4moe_layer_create(ctypes.byref(c), ctypes.byref(w), None) == ds4.ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """The product has no CPU fallback: without the compiled library the
    binding raises instead of computing anything."""
    import pytest
    import quantized_moe_expert_top_gb300._binding as B
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libds4moe.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="is missing"):
        B.lib()


def test_binding_checks_tensor_shapes_before_the_call():
    """The C ABI takes bare pointers, so the binding checks every tensor's
    shape, dtype, contiguity and device before handing its pointer over."""
    import pytest
    import torch
    import quantized_moe_expert_top_gb300._binding as B
    ok = torch.zeros(4, 256, dtype=torch.bfloat16)
    B.check_tensor(ok, "x", (4, 256), torch.bfloat16, on_cuda=False)
    bad = [
        (torch.zeros(4, 256, dtype=torch.float32), "must be torch.bfloat16"),       # dtype
        (torch.zeros(3, 256, dtype=torch.bfloat16), "must have shape"),             # too few rows
        (torch.zeros(4, 128, dtype=torch.bfloat16), "must have shape"),             # too few columns
        (torch.zeros(256, 4, dtype=torch.bfloat16).t(), "must be contiguous"),     # strided view
        ([0.0] * 1024, "must be a torch.Tensor"),
    ]
    for t, msg in bad:
        with pytest.raises(ValueError, match=msg):
            B.check_tensor(t, "x", (4, 256), torch.bfloat16, on_cuda=False)
    with pytest.raises(ValueError, match="current CUDA device"):  # a host tensor where device memory is needed
        B.check_tensor(ok, "x", (4, 256), torch.bfloat16, on_cuda=True)
    with pytest.raises(ValueError, match="2-D"):
        B._rows(torch.zeros(1024, dtype=torch.bfloat16), "x")


def test_expected_weight_shapes_match_the_generators():
    import synth
    import quantized_moe_expert_top_gb300._binding as B
    for down in ("mxfp4", "q2k"):
        wl = synth.Workload("shapes_" + down, 2, 256, 3, 256, 2, 1, 1, "normal", down)
        W = {**synth.make_layer_weights(wl), **synth.make_dense_weights(wl, 64)}
        want = B.expected_weight_shapes(wl.d, wl.E, wl.f, down, 64)
        assert {n: tuple(t.shape) for n, t in W.items()} == {n: want[n] for n in W}


def test_layer_calls_check_before_reaching_the_library(monkeypatch):
    """Layer.forward_host / forward hand their pointers to the library only
    after the checks pass (a fake library records the calls; no GPU)."""
    import pytest
    import torch
    import quantized_moe_expert_top_gb300._binding as B
    calls = []

    class FakeLib:
        def ds4moe_forward_host(self, *a):
            calls.append("forward_host")
            return B.OK

        def ds4moe_forward(self, *a):
            calls.append("forward")
            return B.OK

    class FakeStream:
        cuda_stream = 0

    monkeypatch.setattr(B, "lib", lambda: FakeLib())
    layer = object.__new__(B.Layer)
    layer._h = None
    layer.cfg = B.Config()
    layer.cfg.d_model, layer.cfg.n_experts = 256, 8
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    lg = torch.zeros(4, 8, dtype=torch.float32)
    out = torch.zeros(4, 256, dtype=torch.float32)
    layer.forward_host(x, lg, out, stream=FakeStream())
    assert calls == ["forward_host"]
    for args in ((x, torch.zeros(3, 8), out), (x, lg, torch.zeros(4, 128)), (x.float(), lg, out)):
        with pytest.raises(ValueError):
            layer.forward_host(*args, stream=FakeStream())
    with pytest.raises(ValueError, match="current CUDA device"):
        layer.forward(x, lg, out, stream=FakeStream())
    assert calls == ["forward_host"]
