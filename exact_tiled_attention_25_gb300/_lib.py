"""ctypes view of libattn_gb300.so (the C ABI declared in include/attn_gb300.h).

Loading never falls back to anything: if the library is missing or fails to
load, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

c_int = ctypes.c_int
c_float = ctypes.c_float
c_size_t = ctypes.c_size_t
c_void_p = ctypes.c_void_p
c_char_p = ctypes.c_char_p

# name -> (restype, argtypes); mirrors include/attn_gb300.h
SIGNATURES = {
    "attn_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                         c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_void_p]),
    "attn_fwd_schedule": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                  c_void_p]),
    "attn_fwd_gqa": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_void_p]),
    "attn_fwd_varlen": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                                c_void_p]),
    "attn_bwd_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
    "attn_bwd_gqa": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                             c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_void_p]),
    "attn_bwd_varlen_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "attn_bwd_varlen": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p,
                                c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                                c_void_p]),
    "attn_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                         c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                         c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_void_p]),
    "attn_bwd_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p,
                                 c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_void_p]),
    "attn_fp8_quantize": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "attn_fp8_quantize_gqa": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "attn_fwd_fp8_gqa": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                 c_float, c_void_p]),
    "attn_fp8_quantize_bf16": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "attn_fp8_quantize_varlen": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                         c_int, c_void_p]),
    "attn_fwd_fp8_varlen": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                    c_int, c_int, c_int, c_float, c_void_p]),
    "attn_fp8_quantize_rope": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                       c_void_p]),
    "attn_fp8_quantize_ex": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                     c_int, c_void_p]),
    "attn_decode_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "attn_decode_paged": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_size_t, c_int, c_int, c_int, c_int, c_int,
                                  c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_void_p]),
    "attn_decode_paged_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                      c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                      c_int, c_int, c_float, c_int, c_void_p]),
    "attn_fwd_fp8_schedule": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_float,
                                      c_int, c_void_p]),
    "attn_selftest_exp2": (c_int, [c_void_p, c_void_p, c_void_p, ctypes.c_longlong, c_void_p]),
    "attn_fwd_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_float,
                             c_void_p]),
    "attn_selftest_wait_timeout": (c_int, [ctypes.c_uint, c_void_p]),
    "attn_get_device_status": (c_int, [c_void_p]),
    "attn_status_string": (c_char_p, [c_int]),
    "attn_last_error": (c_char_p, []),
}

_LIB = None


def load(path: str | None = None):
    """Load the library once and declare every entry point's signature."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is not built; run exact_tiled_attention_25_gb300.build.build() "
            "(nvcc for sm_103a is required)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib
