"""ctypes loader for ``lib/libfp8q.so`` and its C signatures (include/fp8q.h).

There is no fallback: if the library has not been built, every call raises.
Build it with ``python -m fp8_scaled_quantization_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libfp8q.so")
HEADER_PATH = os.path.join(os.path.dirname(PKG), "include", "fp8q.h")

_lib = None

c_i32, c_i64, c_f32p, c_vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
c_u64 = ctypes.c_ulonglong

# name -> (restype, argtypes); pointers are passed as integers (c_void_p).
SIGNATURES = {
    "fp8_status_string": (ctypes.c_char_p, [c_i32]),
    "fp8_last_error_message": (ctypes.c_char_p, []),
    "fp8_version": (c_i32, []),
    "fp8_launch_count": (c_u64, []),
    "fp8_wait_timeouts": (c_i32, [c_vp]),
    "fp8_test_drop_tile_copy": (c_i32, [c_i32]),
    "fp8_release_stream_workspace": (c_i32, [c_vp]),
    "fp8_amax": (c_i32, [c_vp, c_i32, c_i64, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "fp8_update_scale_delayed": (c_i32, [c_vp, c_i32, c_i64, c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "fp8_quantize": (c_i32, [c_vp, c_i32, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "fp8_quantize_cast_transpose": (c_i32, [c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "fp8_quantize_block": (c_i32, [c_vp, c_i32, c_i64, c_i64, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "fp8_dequantize": (c_i32, [c_vp, c_i32, c_i64, c_i64, c_vp, c_i32, c_i32, c_vp, c_i32, c_vp]),
    "fp8_quantize_delayed": (c_i32, [c_vp, c_i32, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_i32, c_i64, c_i32, c_i32,
                                     c_vp, c_vp, c_vp]),
    "fp8_quantize_mx": (c_i32, [c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "fp8_dequantize_mx": (c_i32, [c_vp, c_vp, c_i32, c_i64, c_i64, c_vp, c_i32, c_vp]),
    "fp8_block128_scales_to_mx": (c_i32, [c_vp, c_i64, c_i64, c_vp, c_vp, c_vp]),
    "fp8_quantize_current": (c_i32, [c_vp, c_i32, c_i64, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "fp8_quantize_hybrid": (c_i32, [c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_vp, c_i32, c_vp, c_vp, c_i32, c_vp]),
    "fp8_quantize_block_cast_transpose": (c_i32, [c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "fp8_amax_grouped": (c_i32, [c_i32, c_vp, c_vp, c_i32, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "fp8_quantize_grouped": (c_i32, [c_i32, c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "fp8_amax_noalloc": (c_i32, [c_vp, c_i32, c_i64, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp]),
}


class LibraryMissing(RuntimeError):
    pass


def load(path: str = LIB_PATH):
    """Load the library once and attach the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise LibraryMissing(
            f"{path} is missing: the CUDA library must be built first "
            "(python -m fp8_scaled_quantization_gb300.build); there is no CPU fallback")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_entry_points(path: str = HEADER_PATH):
    """Names of the functions declared in include/fp8q.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z0-9_]+)\s*\(", text)))
