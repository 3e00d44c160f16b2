"""CPU oracle for the routed-MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library itself never loads it and
has no CPU fallback.

The arithmetic lives in ``ds4moe_oracle.c`` (plain C, fp64, OpenMP over rows);
this module builds it with gcc and marshals numpy arrays through ctypes.  See
that file's header for the definitions and readings it follows.

Parity pins: tests/test_oracle_pins.py.  The full-size workloads are checked
only through the pinned pieces (codecs, routing, grouping, expert FFN,
combine); nothing here is pinned beyond what those tests cover.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds4moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

ACT_EXACT, ACT_MXFP8, ACT_MXFP8_X_ONLY, ACT_MXFP4 = 0, 1, 2, 3
DOWN_MXFP4, DOWN_Q2K = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no FP contraction so that
    x86 and Arm hosts round identically)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            d, i, u8p, u16p = ctypes.c_double, ctypes.c_int, ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_uint16)
            i32p, dp, fp = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)
            L.ds4o_e2m1.restype = d; L.ds4o_e2m1.argtypes = [ctypes.c_uint]
            L.ds4o_e8m0.restype = d; L.ds4o_e8m0.argtypes = [ctypes.c_uint]
            L.ds4o_half.restype = d; L.ds4o_half.argtypes = [ctypes.c_uint16]
            L.ds4o_bf16.restype = d; L.ds4o_bf16.argtypes = [ctypes.c_uint16]
            L.ds4o_e4m3_decode.restype = d; L.ds4o_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.ds4o_e4m3_encode.restype = ctypes.c_uint8; L.ds4o_e4m3_encode.argtypes = [d]
            L.ds4o_q2k_weight.restype = d; L.ds4o_q2k_weight.argtypes = [u8p, i]
            L.ds4o_mxfp8.restype = None; L.ds4o_mxfp8.argtypes = [dp, i, u8p, u8p]
            L.ds4o_e2m1_encode.restype = ctypes.c_uint8; L.ds4o_e2m1_encode.argtypes = [d]
            L.ds4o_mxfp4_act.restype = None; L.ds4o_mxfp4_act.argtypes = [dp, i, u8p, u8p]
            L.ds4o_route.restype = None; L.ds4o_route.argtypes = [fp, i, i, i, i32p, dp]
            L.ds4o_group.restype = None; L.ds4o_group.argtypes = [i32p, i, i, i, i32p, i32p, i32p, i32p, i32p]
            fwd_args = [i, i, i, i, i, i] + [u8p] * 7 + [u16p, i32p, dp, i, i32p, dp]
            L.ds4o_forward.restype = None; L.ds4o_forward.argtypes = fwd_args
            L.ds4o_forward_dense.restype = None; L.ds4o_forward_dense.argtypes = fwd_args
            L.ds4o_dequant_expert.restype = None
            L.ds4o_dequant_expert.argtypes = [i, i, i, i, i] + [u8p] * 7 + [dp, dp, dp]
            L.ds4o_num_threads.restype = i; L.ds4o_num_threads.argtypes = []
            L.ds4o_router_logits.restype = None
            L.ds4o_router_logits.argtypes = [i, i, u16p, u16p, i, dp]
            L.ds4o_shared_ffn.restype = None
            L.ds4o_shared_ffn.argtypes = [i, i, u16p, u16p, u16p, u16p, i, i32p, dp]
            _lib = L
    return _lib


# ---------------------------------------------------------------- formats
def e2m1(code: int) -> float:
    return lib().ds4o_e2m1(code)


def e8m0(b: int) -> float:
    return lib().ds4o_e8m0(b)


def half(bits: int) -> float:
    return lib().ds4o_half(bits)


def bf16(bits: int) -> float:
    return lib().ds4o_bf16(bits)


def e4m3_encode(v: float) -> int:
    return int(lib().ds4o_e4m3_encode(float(v)))


def e4m3_decode(b: int) -> float:
    return lib().ds4o_e4m3_decode(b)


def e2m1_encode(v: float) -> int:
    return int(lib().ds4o_e2m1_encode(float(v)))


def mxfp4_act(v: np.ndarray):
    """MXFP4 of a 1-D fp64 activation vector (len % 32 == 0) -> (codes uint8,
    one E2M1 code 0..15 per element; scales uint8)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    n = v.size
    assert n % 32 == 0
    codes = np.empty(n, np.uint8)
    scales = np.empty(n // 32, np.uint8)
    lib().ds4o_mxfp4_act(_p(v, ctypes.c_double), n, _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8))
    return codes, scales


def q2k_weight(block: np.ndarray, i: int) -> float:
    block = np.ascontiguousarray(block, dtype=np.uint8)
    assert block.size == 84
    return lib().ds4o_q2k_weight(_p(block, ctypes.c_uint8), i)


def mxfp8(v: np.ndarray):
    """MXFP8 of a 1-D fp64 vector (len % 32 == 0) -> (codes uint8, scales uint8)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    n = v.size
    assert n % 32 == 0
    codes = np.empty(n, np.uint8)
    scales = np.empty(n // 32, np.uint8)
    lib().ds4o_mxfp8(_p(v, ctypes.c_double), n, _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8))
    return codes, scales


# ---------------------------------------------------------------- routing
def route(logits: np.ndarray, k: int):
    """-> (idx int32 [T,k], w float64 [T,k])."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().ds4o_route(_p(logits, ctypes.c_float), T, E, k, _p(idx, ctypes.c_int32), _p(w, ctypes.c_double))
    return idx, w


def group(idx: np.ndarray, E: int) -> dict:
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm_tok = np.empty(T * k, np.int32)
    perm_slot = np.empty(T * k, np.int32)
    inv = np.empty((T, k), np.int32)
    i32 = ctypes.c_int32
    lib().ds4o_group(_p(idx, i32), T, E, k, _p(counts, i32), _p(offsets, i32), _p(perm_tok, i32),
                     _p(perm_slot, i32), _p(inv, i32))
    return {"counts": counts, "offsets": offsets, "perm_tok": perm_tok, "perm_slot": perm_slot, "inv": inv}


# ---------------------------------------------------------------- forward
_EMPTY = np.zeros(16, np.uint8)


def _weights_args(W: dict):
    """Canonical weight dict (numpy uint8 arrays) -> 7 pointers + down format."""
    def arr(name):
        a = W.get(name)
        if a is None:
            return _EMPTY
        return np.ascontiguousarray(a, dtype=np.uint8)
    keep = [arr(n) for n in ("gate_codes", "gate_scales", "up_codes", "up_scales",
                              "down_codes", "down_scales", "down_q2k")]
    down_fmt = DOWN_Q2K if W.get("down_q2k") is not None else DOWN_MXFP4
    return keep, down_fmt


def _forward(fn, dims: dict, W: dict, x_bf16_bits: np.ndarray, idx: np.ndarray, w: np.ndarray,
             tokens, act_mode: int) -> np.ndarray:
    keep, down_fmt = _weights_args(W)
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n = tokens.size
    out = np.empty((n, dims["d"]), np.float64)
    ptrs = [_p(a, ctypes.c_uint8) for a in keep]
    fn(dims["d"], dims["E"], dims["f"], dims["k"], down_fmt, act_mode, *ptrs,
       _p(x, ctypes.c_uint16), _p(idx, ctypes.c_int32), _p(w, ctypes.c_double), n,
       _p(tokens, ctypes.c_int32), _p(out, ctypes.c_double))
    return out


def forward(dims, W, x_bf16_bits, idx, w, tokens, act_mode=ACT_EXACT) -> np.ndarray:
    """Routed layer output (fp64) for the listed tokens: [len(tokens), d]."""
    return _forward(lib().ds4o_forward, dims, W, x_bf16_bits, idx, w, tokens, act_mode)


def forward_dense(dims, W, x_bf16_bits, idx, w, tokens, act_mode=ACT_EXACT) -> np.ndarray:
    """Brute force over all experts with a (0 | w) mask: [len(tokens), d]."""
    return _forward(lib().ds4o_forward_dense, dims, W, x_bf16_bits, idx, w, tokens, act_mode)


def dequant_expert(dims, W, e: int):
    """Decoded fp64 weights of expert e: (wg [f,d], wu [f,d], wd [d,f])."""
    keep, down_fmt = _weights_args(W)
    d, f = dims["d"], dims["f"]
    wg = np.empty((f, d)); wu = np.empty((f, d)); wd = np.empty((d, f))
    ptrs = [_p(a, ctypes.c_uint8) for a in keep]
    lib().ds4o_dequant_expert(d, dims["E"], f, down_fmt, e, *ptrs,
                              _p(wg, ctypes.c_double), _p(wu, ctypes.c_double), _p(wd, ctypes.c_double))
    return wg, wu, wd


# ---------------------------------------------------------------- router and shared expert
def router_logits(wr_bits: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """fp64 router logits [T, E] of bf16 weights wr [E, d] and bf16 x [T, d]."""
    wr = np.ascontiguousarray(wr_bits, dtype=np.uint16)
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    E, d = wr.shape
    T = x.shape[0]
    out = np.empty((T, E), np.float64)
    lib().ds4o_router_logits(d, E, _p(wr, ctypes.c_uint16), _p(x, ctypes.c_uint16), T, _p(out, ctypes.c_double))
    return out


def shared_ffn(wg_bits, wu_bits, wd_bits, x_bits, tokens) -> np.ndarray:
    """Shared-expert output (fp64) for the listed tokens: [len(tokens), d]."""
    wg = np.ascontiguousarray(wg_bits, dtype=np.uint16)
    wu = np.ascontiguousarray(wu_bits, dtype=np.uint16)
    wd = np.ascontiguousarray(wd_bits, dtype=np.uint16)
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    fs, d = wg.shape
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    y = np.empty((tokens.size, d), np.float64)
    lib().ds4o_shared_ffn(d, fs, _p(wg, ctypes.c_uint16), _p(wu, ctypes.c_uint16), _p(wd, ctypes.c_uint16),
                          _p(x, ctypes.c_uint16), tokens.size, _p(tokens, ctypes.c_int32), _p(y, ctypes.c_double))
    return y


def num_threads() -> int:
    return int(lib().ds4o_num_threads())
