"""ctypes binding of libds4moe.so (include/ds4moe.h).

Argument marshalling only: torch tensors supply device memory and
``data_ptr()``; torch streams supply the ``cudaStream_t``.  Every step of the
layer runs in the library's CUDA kernels; there is no Python or CPU fallback,
and loading fails loudly when the compiled library is missing.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libds4moe.so")
HEADER_PATH = os.path.join(_HERE, "..", "include", "ds4moe.h")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_OOM = -4
ERR_TOO_MANY_TOKENS = -5
ERR_DEVICE_TIMEOUT = -6

DOWN_MXFP4, DOWN_Q2K = 0, 1
PATH_AUTO, PATH_DECODE, PATH_PREFILL, PATH_DECODE_MMA = 0, 1, 2, 3
_PATHS = {"auto": PATH_AUTO, "decode": PATH_DECODE, "prefill": PATH_PREFILL, "decode_mma": PATH_DECODE_MMA}
_DOWN = {"mxfp4": DOWN_MXFP4, "q2k": DOWN_Q2K}


class Ds4moeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "d_model", "n_experts", "d_ff", "top_k", "max_tokens", "down_format",
        "decode_max_tokens", "force_path", "debug_fault", "wait_timeout_ms", "has_router", "d_ff_shared")]


class WeightPtrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "gate_codes", "gate_scales", "up_codes", "up_scales", "down_codes", "down_scales",
        "router", "shared_gate", "shared_up", "shared_down")]

_DENSE = ("router", "shared_gate", "shared_up", "shared_down")


_lib = None


def header_functions() -> list:
    """Names of the functions declared in include/ds4moe.h."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"\b(ds4moe_[a-z_]+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python quantized_moe_expert_top_gb300/_builder.py` (or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        L.ds4moe_config_default.restype = None
        L.ds4moe_config_default.argtypes = [ctypes.POINTER(Config)]
        L.ds4moe_layer_create.restype = ctypes.c_int
        L.ds4moe_layer_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(WeightPtrs), ctypes.POINTER(vp)]
        L.ds4moe_forward.restype = ctypes.c_int
        L.ds4moe_forward.argtypes = [vp, vp, vp, vp, i32, vp]
        L.ds4moe_forward_x.restype = ctypes.c_int
        L.ds4moe_forward_x.argtypes = [vp, vp, vp, i32, vp]
        L.ds4moe_get_logits.restype = ctypes.c_int
        L.ds4moe_get_logits.argtypes = [vp, vp, vp]
        L.ds4moe_forward_host.restype = ctypes.c_int
        L.ds4moe_forward_host.argtypes = [vp, vp, vp, vp, i32, vp]
        L.ds4moe_get_routing.restype = ctypes.c_int
        L.ds4moe_get_routing.argtypes = [vp, vp, vp, vp, vp, vp]
        L.ds4moe_get_status.restype = ctypes.c_int
        L.ds4moe_get_status.argtypes = [vp]
        L.ds4moe_path_for.restype = ctypes.c_int
        L.ds4moe_path_for.argtypes = [vp, i32]
        L.ds4moe_launches_per_forward.restype = ctypes.c_int
        L.ds4moe_launches_per_forward.argtypes = [vp, i32]
        L.ds4moe_set_kernel_timing.restype = ctypes.c_int
        L.ds4moe_set_kernel_timing.argtypes = [vp, ctypes.c_int]
        L.ds4moe_kernel_times.restype = ctypes.c_int
        L.ds4moe_kernel_times.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.c_int]
        L.ds4moe_kernel_name.restype = ctypes.c_char_p
        L.ds4moe_kernel_name.argtypes = [vp, i32, ctypes.c_int]
        L.ds4moe_get_act_codes.restype = ctypes.c_int
        L.ds4moe_get_act_codes.argtypes = [vp, i32, vp, vp, vp]
        L.ds4moe_route_noalloc.restype = ctypes.c_int
        L.ds4moe_route_noalloc.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
        L.ds4moe_status_string.restype = ctypes.c_char_p
        L.ds4moe_status_string.argtypes = [ctypes.c_int]
        L.ds4moe_destroy.restype = None
        L.ds4moe_destroy.argtypes = [vp]
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().ds4moe_status_string(code).decode()


def default_config() -> Config:
    c = Config()
    lib().ds4moe_config_default(ctypes.byref(c))
    return c


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def check_tensor(t, name: str, shape: tuple, dtype: torch.dtype, on_cuda: bool) -> None:
    """Raise ValueError unless t is a contiguous tensor of exactly this shape
    and dtype, on the current CUDA device (on_cuda) or on the host.  The C ABI
    takes bare pointers, so a smaller buffer than the call implies would be
    read or written past its end by the kernels."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if on_cuda:
        if not t.is_cuda or t.device.index != torch.cuda.current_device():
            raise ValueError(f"{name} must be on the current CUDA device")
    elif t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")


def expected_weight_shapes(d: int, E: int, f: int, down: str, fs: int = 0) -> dict:
    """Shapes of the stored weight tensors a layer of these sizes reads."""
    shapes = {"gate_codes": (E, f, d // 2), "gate_scales": (E, f, d // 32),
              "up_codes": (E, f, d // 2), "up_scales": (E, f, d // 32),
              "router": (E, d), "shared_gate": (fs, d), "shared_up": (fs, d), "shared_down": (d, fs)}
    if down == "q2k":
        shapes["down_q2k"] = (E, d, f // 256, 84)
    else:
        shapes["down_codes"] = (E, d, f // 2)
        shapes["down_scales"] = (E, d, f // 32)
    return shapes


def _rows(t, name: str) -> int:
    if not isinstance(t, torch.Tensor) or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D tensor [T, ...]")
    return t.shape[0]


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def route_noalloc(logits: torch.Tensor, k: int, stream=None) -> dict:
    """Routing through ds4moe_route_noalloc (no device allocation inside the
    library; the output tensors are allocated here by torch)."""
    T = _rows(logits, "logits")
    E = logits.shape[1]
    check_tensor(logits, "logits", (T, E), torch.float32, on_cuda=True)
    dev = logits.device
    r = {"topk_idx": torch.empty(max(T, 1), k, dtype=torch.int32, device=dev),
         "topk_w": torch.empty(max(T, 1), k, dtype=torch.float32, device=dev),
         "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
         "perm_tok": torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)}
    rc = lib().ds4moe_route_noalloc(_ptr(logits), T, E, k, _ptr(r["topk_idx"]), _ptr(r["topk_w"]),
                                    _ptr(r["offsets"]), _ptr(r["perm_tok"]), _stream_handle(stream))
    if rc != OK:
        raise Ds4moeError(rc, "ds4moe_route_noalloc")
    r["topk_idx"], r["topk_w"], r["perm_tok"] = r["topk_idx"][:T], r["topk_w"][:T], r["perm_tok"][:T * k]
    return r


class Layer:
    """One routed-MoE expert layer owned by the library.

    ``weights`` holds the canonical stored tensors on the current CUDA device
    (uint8): gate_codes/up_codes [E,f,d/2], gate_scales/up_scales [E,f,d/32],
    and either down_codes [E,d,f/2] + down_scales [E,d,f/32] (MXFP4) or
    down_q2k [E,d,f/256,84] (Q2_K); optionally, in bf16, router [E,d] and a
    shared expert shared_gate/shared_up [fs,d], shared_down [d,fs].  The
    library copies them; the caller may free them after construction."""

    def __init__(self, d_model: int, n_experts: int, d_ff: int, top_k: int, max_tokens: int,
                 weights: dict, decode_max_tokens: int = 64, force_path: str = "auto",
                 debug_fault: int = 0, wait_timeout_ms: int = 2000):
        self._h = None
        down = "q2k" if weights.get("down_q2k") is not None else "mxfp4"
        c = default_config()
        c.d_model, c.n_experts, c.d_ff, c.top_k = d_model, n_experts, d_ff, top_k
        c.max_tokens = max_tokens
        c.down_format = _DOWN[down]
        c.decode_max_tokens = decode_max_tokens
        c.force_path = _PATHS[force_path]
        c.debug_fault = debug_fault
        c.wait_timeout_ms = wait_timeout_ms
        c.has_router = 1 if weights.get("router") is not None else 0
        c.d_ff_shared = weights["shared_gate"].shape[0] if weights.get("shared_gate") is not None else 0
        self.cfg = c
        self.down = down
        shapes = expected_weight_shapes(d_model, n_experts, d_ff, down, c.d_ff_shared)
        sizes_ok = d_model % 128 == 0 and d_ff % (256 if down == "q2k" else 128) == 0 and c.d_ff_shared % 32 == 0
        for name, t in weights.items():
            if t is None:
                continue
            if name not in shapes:
                raise ValueError(f"unknown weight {name}")
            want = torch.bfloat16 if name in _DENSE else torch.uint8
            # sizes the library rejects are left to its own status code
            check_tensor(t, f"weight {name}", shapes[name] if sizes_ok else tuple(t.shape), want, on_cuda=True)
        w = WeightPtrs()
        w.gate_codes = weights["gate_codes"].data_ptr()
        w.gate_scales = weights["gate_scales"].data_ptr()
        w.up_codes = weights["up_codes"].data_ptr()
        w.up_scales = weights["up_scales"].data_ptr()
        if down == "q2k":
            w.down_codes = weights["down_q2k"].data_ptr()
            w.down_scales = None
        else:
            w.down_codes = weights["down_codes"].data_ptr()
            w.down_scales = weights["down_scales"].data_ptr()
        for name in _DENSE:
            if weights.get(name) is not None:
                setattr(w, name, weights[name].data_ptr())
        h = ctypes.c_void_p()
        rc = lib().ds4moe_layer_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h))
        if rc != OK:
            raise Ds4moeError(rc, "ds4moe_layer_create")
        self._h = h
        self._last_T = 0

    # ------------------------------------------------------------------
    def forward(self, x: torch.Tensor, logits: torch.Tensor, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
        """Enqueue one forward pass (asynchronous on `stream`)."""
        T, d, E = _rows(x, "x"), self.cfg.d_model, self.cfg.n_experts
        if out is None:
            out = torch.empty(T, d, dtype=torch.float32, device=x.device)
        check_tensor(x, "x", (T, d), torch.bfloat16, on_cuda=True)
        check_tensor(logits, "logits", (T, E), torch.float32, on_cuda=True)
        check_tensor(out, "out", (T, d), torch.float32, on_cuda=True)
        rc = lib().ds4moe_forward(self._h, _ptr(x), _ptr(logits), _ptr(out), T, _stream_handle(stream))
        if rc != OK:
            raise Ds4moeError(rc, "ds4moe_forward")
        self._last_T = T
        return out

    def forward_x(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """The layer from x alone: router logits, routed experts, shared expert."""
        T, d = _rows(x, "x"), self.cfg.d_model
        if out is None:
            out = torch.empty(T, d, dtype=torch.float32, device=x.device)
        check_tensor(x, "x", (T, d), torch.bfloat16, on_cuda=True)
        check_tensor(out, "out", (T, d), torch.float32, on_cuda=True)
        rc = lib().ds4moe_forward_x(self._h, _ptr(x), _ptr(out), T, _stream_handle(stream))
        if rc != OK:
            raise Ds4moeError(rc, "ds4moe_forward_x")
        self._last_T = T
        return out

    def logits(self, stream=None) -> torch.Tensor:
        """Router logits of the last forward_x call [T, E] (fp32, device)."""
        dev = torch.device("cuda", torch.cuda.current_device())
        r = torch.empty(self._last_T, self.cfg.n_experts, dtype=torch.float32, device=dev)
        rc = lib().ds4moe_get_logits(self._h, _ptr(r), _stream_handle(stream))
        if rc != OK:
            raise Ds4moeError(rc, "ds4moe_get_logits")
        return r

    def forward_host(self, x: torch.Tensor, logits: torch.Tensor, out: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
        """Forward pass on host tensors (copies in, runs, copies out, synchronises)."""
        T, d, E = _rows(x, "x"), self.cfg.d_model, self.cfg.n_experts
        if out is None:
            out = torch.empty(T, d, dtype=torch.float32, pin_memory=True)
        check_tensor(x, "x", (T, d), torch.bfloat16, on_cuda=False)
        check_tensor(logits, "logits", (T, E), torch.float32, on_cuda=False)
        check_tensor(out, "out", (T, d), torch.float32, on_cuda=False)
        rc = lib().ds4moe_forward_host(self._h, _ptr(x), _ptr(logits), _ptr(out), T, _stream_handle(stream))
        if rc != OK:
            raise Ds4moeError(rc, "ds4moe_forward_host")
        self._last_T = T
        return out

    def routing(self, stream=None) -> dict:
        """Routing tables of the last forward (device tensors)."""
        T, k, E = self._last_T, self.cfg.top_k, self.cfg.n_experts
        dev = torch.device("cuda", torch.cuda.current_device())
        r = {"topk_idx": torch.empty(T, k, dtype=torch.int32, device=dev),
             "topk_w": torch.empty(T, k, dtype=torch.float32, device=dev),
             "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
             "perm_tok": torch.empty(T * k, dtype=torch.int32, device=dev)}
        rc = lib().ds4moe_get_routing(self._h, _ptr(r["topk_idx"]), _ptr(r["topk_w"]), _ptr(r["offsets"]),
                                      _ptr(r["perm_tok"]), _stream_handle(stream))
        if rc != OK:
            raise Ds4moeError(rc, "ds4moe_get_routing")
        return r

    def act_codes(self, which: str = "x", stream=None) -> dict:
        """MXFP8 activation rows of the last forward (diagnostics): x or h
        codes [T*k*S, K] and scale bytes [T*k*S, K/32] in token order of the
        routed pairs, S rows per pair (1 on PREFILL, 2 = hi, lo on DECODE_MMA)."""
        T, k = self._last_T, self.cfg.top_k
        K = self.cfg.d_model if which == "x" else self.cfg.d_ff
        dev = torch.device("cuda", torch.cuda.current_device())
        codes = torch.empty(max(2 * T * k, 1), K, dtype=torch.uint8, device=dev)
        scales = torch.empty(max(2 * T * k, 1), K // 32, dtype=torch.uint8, device=dev)
        n = lib().ds4moe_get_act_codes(self._h, 0 if which == "x" else 1, _ptr(codes), _ptr(scales),
                                       _stream_handle(stream))
        if n < 0:
            raise Ds4moeError(n, "ds4moe_get_act_codes")
        return {"split": n, "codes": codes[:T * k * n], "scales": scales[:T * k * n]}

    def status(self) -> int:
        return lib().ds4moe_get_status(self._h)

    def path_for(self, T: int) -> int:
        return lib().ds4moe_path_for(self._h, T)

    def launches_per_forward(self, T: int) -> int:
        return lib().ds4moe_launches_per_forward(self._h, T)

    def set_kernel_timing(self, enable: bool):
        rc = lib().ds4moe_set_kernel_timing(self._h, 1 if enable else 0)
        if rc != OK:
            raise Ds4moeError(rc, "ds4moe_set_kernel_timing")

    def kernel_times(self) -> dict:
        """{kernel name: ms} of the most recent forward (timing must be on)."""
        buf = (ctypes.c_float * 12)()
        n = lib().ds4moe_kernel_times(self._h, buf, 12)
        if n < 0:
            raise Ds4moeError(n, "ds4moe_kernel_times")
        return {lib().ds4moe_kernel_name(self._h, self._last_T, i).decode(): float(buf[i]) for i in range(n)}

    def close(self):
        if self._h is not None:
            lib().ds4moe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
