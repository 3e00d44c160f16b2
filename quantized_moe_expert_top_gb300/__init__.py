"""ds4moe -- the routed-MoE expert layer with 4-bit block-scaled (MXFP4) experts
and a Q2_K-style 2-bit down-projection variant, as hand-written CUDA for GB300
(sm_103a) behind a C ABI (include/ds4moe.h).

Python sees a thin ctypes binding (:class:`Layer`); the compiled library is
built in-tree by :func:`build`.
"""
from ._binding import (  # noqa: F401
    Config, Ds4moeError, Layer, WeightPtrs, default_config, header_functions, lib, route_noalloc, status_string,
    OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_TOO_MANY_TOKENS, ERR_DEVICE_TIMEOUT,
    DOWN_MXFP4, DOWN_Q2K, PATH_AUTO, PATH_DECODE, PATH_PREFILL, PATH_DECODE_MMA, LIB_PATH,
)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libds4moe.so for sm_103a (no-op when up to date)."""
    from ._builder import build as _build
    return _build(force=force, verbose=verbose)
