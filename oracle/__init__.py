"""CPU oracle for FP8 scaled quantization -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never touches it, and this package never imports the product.

The arithmetic lives in ``fp8_oracle.c`` (plain scalar C, one element at a
time).  This module only compiles it, loads it with ctypes and marshals numpy
arrays.  For large inputs it may run the same C loop on disjoint row ranges
in threads; every function below is an element-wise map or an exact maximum,
so the result does not depend on the split.

Array conventions: BF16 data is carried as ``numpy.uint16`` bit patterns,
fp32 as ``numpy.float32``, FP8 codes as ``numpy.uint8``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

E4M3, E5M2 = 0, 1
BF16, FP32 = 0, 1
ALGO_MAX, ALGO_MOST_RECENT = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB = os.path.join(_HERE, "libfp8_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE fp32: no contraction, no fast math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        vp, u8 = ctypes.c_void_p, ctypes.c_uint8
        L.oref_decode_f64.argtypes, L.oref_decode_f64.restype = [u8, i32], f64
        L.oref_decode.argtypes, L.oref_decode.restype = [u8, i32], f32
        L.oref_max_finite.argtypes, L.oref_max_finite.restype = [i32], f64
        L.oref_min_normal.argtypes, L.oref_min_normal.restype = [i32], f64
        L.oref_format_stats.argtypes = [i32, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(f64)]
        L.oref_format_stats.restype = None
        L.oref_encode_saturating.argtypes, L.oref_encode_saturating.restype = [f32, i32], u8
        L.oref_quantize_element.argtypes = [f32, f32, i32, ctypes.POINTER(i32)]
        L.oref_quantize_element.restype = u8
        L.oref_bf16_to_f32.argtypes, L.oref_bf16_to_f32.restype = [ctypes.c_uint16], f32
        L.oref_f32_to_bf16.argtypes, L.oref_f32_to_bf16.restype = [f32], ctypes.c_uint16
        L.oref_amax.argtypes, L.oref_amax.restype = [vp, i32, i64], f32
        L.oref_compute_scale.argtypes = [f32, i32, i32, ctypes.POINTER(f32), ctypes.POINTER(f32)]
        L.oref_compute_scale.restype = None
        L.oref_quantize.argtypes, L.oref_quantize.restype = [vp, i32, i64, i32, f32, vp], ctypes.c_uint64
        L.oref_cast_transpose.argtypes = [vp, i32, i64, i64, i32, f32, vp, vp]
        L.oref_cast_transpose.restype = None
        L.oref_update_delayed.argtypes = [vp, i32, i64, vp, i32, i32, i32,
                                          ctypes.POINTER(f32), ctypes.POINTER(f32)]
        L.oref_update_delayed.restype = None
        L.oref_quantize_block.argtypes = [vp, i32, i64, i64, i32, i32, i32, vp, vp]
        L.oref_quantize_block.restype = None
        L.oref_dequantize.argtypes = [vp, i32, i64, i64, vp, i32, i32, vp, i32]
        L.oref_dequantize.restype = None
        L.oref_e8m0_decode.argtypes, L.oref_e8m0_decode.restype = [u8], f64
        L.oref_quantize_mx.argtypes = [vp, i32, i64, i64, i32, vp, vp]
        L.oref_quantize_mx.restype = None
        L.oref_dequantize_mx.argtypes = [vp, vp, i64, i64, i32, vp, i32]
        L.oref_dequantize_mx.restype = None
        L.oref_block128_scales_to_mx.argtypes = [vp, i64, i64, vp]
        L.oref_block128_scales_to_mx.restype = i64
        L.oref_quantize_hybrid.argtypes = [vp, i32, i64, i64, i32, f32, i32, f32, i32, vp, vp]
        L.oref_quantize_hybrid.restype = None
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _dtype_of(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return BF16
    if x.dtype == np.float32:
        return FP32
    raise TypeError(f"oracle input must be uint16 (bf16 bits) or float32, got {x.dtype}")


def _chunks(n: int, threads: int, align: int = 1):
    """Split [0, n) into at most `threads` ranges whose starts are multiples of `align`."""
    if n <= 0:
        return [(0, 0)]
    threads = max(1, min(threads, (n + align - 1) // align))
    step = -(-n // threads)
    step = -(-step // align) * align
    return [(s, min(n, s + step)) for s in range(0, n, step)]


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# --------------------------------------------------------------------------- formats

def decode(codes, fmt: int) -> np.ndarray:
    """Exact fp32 value of each code."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    L = lib()
    table = np.array([L.oref_decode(i, fmt) for i in range(256)], dtype=np.float32)
    return table[c]


def decode_f64(code: int, fmt: int) -> float:
    return lib().oref_decode_f64(code, fmt)


def max_finite(fmt: int) -> float:
    return lib().oref_max_finite(fmt)


def min_normal(fmt: int) -> float:
    return lib().oref_min_normal(fmt)


def format_stats(fmt: int):
    b, e = ctypes.c_int(), ctypes.c_int()
    m = ctypes.c_double()
    lib().oref_format_stats(fmt, ctypes.byref(b), ctypes.byref(e), ctypes.byref(m))
    return b.value, e.value, m.value


def encode_saturating(p, fmt: int) -> np.ndarray:
    p = np.ascontiguousarray(p, dtype=np.float32).ravel()
    L = lib()
    return np.array([L.oref_encode_saturating(float(v), fmt) for v in p], dtype=np.uint8)


def bf16_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    L = lib()
    return np.array([L.oref_bf16_to_f32(int(v)) for v in b], dtype=np.float32)


def f32_to_bf16(vals) -> np.ndarray:
    v = np.ascontiguousarray(vals, dtype=np.float32).ravel()
    L = lib()
    return np.array([L.oref_f32_to_bf16(float(a)) for a in v], dtype=np.uint16)


# --------------------------------------------------------------------------- scaling

def amax(x: np.ndarray, threads: int = 1) -> np.float32:
    """max |x| (NaN propagates as the canonical quiet NaN; empty -> 0)."""
    x = np.ascontiguousarray(x).ravel()
    dt = _dtype_of(x)
    L = lib()
    parts = _chunks(x.size, threads)

    def run(se):
        s, e = se
        return np.float32(L.oref_amax(_ptr(x) + s * x.itemsize, dt, e - s))

    if len(parts) == 1:
        return run(parts[0])
    with ThreadPoolExecutor(len(parts)) as ex:
        vals = list(ex.map(run, parts))
    # exact maximum of the chunk maxima (NaN wins)
    for v in vals:
        if np.isnan(v):
            return v
    return np.float32(max(vals))


def compute_scale(amax_value, fmt: int, margin: int = 0):
    s, si = ctypes.c_float(), ctypes.c_float()
    lib().oref_compute_scale(float(np.float32(amax_value)), fmt, margin, ctypes.byref(s), ctypes.byref(si))
    return np.float32(s.value), np.float32(si.value)


def quantize(x: np.ndarray, fmt: int, scale, threads: int = 1):
    """Per-tensor quantize. Returns (codes uint8 shaped like x, saturated count)."""
    shape = x.shape
    x = np.ascontiguousarray(x).ravel()
    dt = _dtype_of(x)
    q = np.empty(x.size, dtype=np.uint8)
    L = lib()
    sc = float(np.float32(scale))

    def run(se):
        s, e = se
        return L.oref_quantize(_ptr(x) + s * x.itemsize, dt, e - s, fmt, sc, _ptr(q) + s)

    parts = _chunks(x.size, threads)
    if len(parts) == 1:
        sat = run(parts[0])
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            sat = sum(ex.map(run, parts))
    return q.reshape(shape), int(sat)


def quantize_element(x: float, scale: float, fmt: int):
    s = ctypes.c_int()
    c = lib().oref_quantize_element(float(np.float32(x)), float(np.float32(scale)), fmt, ctypes.byref(s))
    return c, s.value


def cast_transpose(x: np.ndarray, fmt: int, scale, threads: int = 1):
    """Rowwise [rows, cols] and columnwise [cols, rows] codes under one scale."""
    assert x.ndim == 2
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    dt = _dtype_of(x)
    q_row = np.empty((rows, cols), dtype=np.uint8)
    q_col = np.empty((cols, rows), dtype=np.uint8)
    L = lib()
    sc = float(np.float32(scale))

    def run(se):
        s, e = se
        part_col = np.empty((cols, e - s), dtype=np.uint8)
        L.oref_cast_transpose(_ptr(x) + s * cols * x.itemsize, dt, e - s, cols, fmt, sc,
                              _ptr(q_row) + s * cols, _ptr(part_col))
        q_col[:, s:e] = part_col

    parts = _chunks(rows, threads)
    if len(parts) == 1:
        run(parts[0])
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(run, parts))
    return q_row, q_col


def update_delayed(history: np.ndarray, step: int, new_amax, algo: int, fmt: int, margin: int = 0):
    """In-place delayed-scaling update of a float32 history; returns (scale, scale_inv)."""
    assert history.dtype == np.float32 and history.flags["C_CONTIGUOUS"]
    s, si = ctypes.c_float(), ctypes.c_float()
    if new_amax is None:
        na = None
    else:
        na_arr = np.array([new_amax], dtype=np.float32)
        na = _ptr(na_arr)
    lib().oref_update_delayed(_ptr(history), history.size, step, na, algo, fmt, margin,
                              ctypes.byref(s), ctypes.byref(si))
    return np.float32(s.value), np.float32(si.value)


def quantize_block(x: np.ndarray, br: int, bc: int, fmt: int, threads: int = 1):
    """Block-scaled quantize. Returns (codes [rows, cols], scale_inv [ceil(r/br), ceil(c/bc)])."""
    assert x.ndim == 2
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    dt = _dtype_of(x)
    nbr, nbc = -(-rows // br), -(-cols // bc)
    q = np.empty((rows, cols), dtype=np.uint8)
    si = np.empty((nbr, nbc), dtype=np.float32)
    L = lib()

    def run(se):
        s, e = se  # row range, aligned to whole block rows
        L.oref_quantize_block(_ptr(x) + s * cols * x.itemsize, dt, e - s, cols, br, bc, fmt,
                              _ptr(q) + s * cols, _ptr(si) + (s // br) * nbc * 4)

    parts = _chunks(rows, threads, align=br)
    if len(parts) == 1:
        run(parts[0])
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(run, parts))
    return q, si


def dequantize(q: np.ndarray, fmt: int, scale_inv, br: int = 0, bc: int = 0, out_dt: int = BF16,
               threads: int = 1) -> np.ndarray:
    """y = decode(q) * scale_inv (fp32), then BF16 (uint16 bits) or fp32 output."""
    q2 = np.ascontiguousarray(q)
    if q2.ndim == 1:
        q2 = q2.reshape(1, -1)
    rows, cols = q2.shape
    si = np.ascontiguousarray(scale_inv, dtype=np.float32)
    y = np.empty((rows, cols), dtype=np.uint16 if out_dt == BF16 else np.float32)
    L = lib()
    nbc = -(-cols // bc) if bc > 0 else 0

    def run(se):
        s, e = se
        si_off = (s // br) * nbc * 4 if br > 0 else 0
        L.oref_dequantize(_ptr(q2) + s * cols, fmt, e - s, cols, _ptr(si) + si_off, br, bc,
                          _ptr(y) + s * cols * y.itemsize, out_dt)

    parts = _chunks(rows, threads, align=br if br > 0 else 1)
    if len(parts) == 1:
        run(parts[0])
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(run, parts))
    return y.reshape(q.shape)


# --------------------------------------------------------------------------- MXFP8

MX_BLOCK = 32


def e8m0_decode(code: int) -> float:
    return lib().oref_e8m0_decode(code)


def quantize_mx(x: np.ndarray, fmt: int, threads: int = 1):
    """Rowwise MX quantize of [rows, cols]: (codes [rows, cols], E8M0 scales [rows, ceil(cols/32)])."""
    assert x.ndim == 2
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    dt = _dtype_of(x)
    nb = -(-cols // MX_BLOCK)
    q = np.empty((rows, cols), dtype=np.uint8)
    sc = np.empty((rows, nb), dtype=np.uint8)
    L = lib()

    def run(se):
        s, e = se
        L.oref_quantize_mx(_ptr(x) + s * cols * x.itemsize, dt, e - s, cols, fmt, _ptr(q) + s * cols,
                           _ptr(sc) + s * nb)

    parts = _chunks(rows, threads)
    if len(parts) == 1:
        run(parts[0])
    else:
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(run, parts))
    return q, sc


def dequantize_mx(q: np.ndarray, scales: np.ndarray, fmt: int, out_dt: int = BF16) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, cols = q.shape
    y = np.empty((rows, cols), dtype=np.uint16 if out_dt == BF16 else np.float32)
    lib().oref_dequantize_mx(_ptr(q), _ptr(sc), rows, cols, fmt, _ptr(y), out_dt)
    return y


def block128_scales_to_mx(scale_inv: np.ndarray, rows: int, cols: int):
    """E8M0 [rows, ceil(cols/32)] scales from 128x128 fp32 scale_inv; returns (scales, non-power-of-two blocks)."""
    si = np.ascontiguousarray(scale_inv, dtype=np.float32)
    out = np.empty((rows, -(-cols // MX_BLOCK)), dtype=np.uint8)
    bad = lib().oref_block128_scales_to_mx(_ptr(si), rows, cols, _ptr(out))
    return out, int(bad)


# --------------------------------------------------------------------------- hybrid

SRC_ORIGINAL, SRC_ROWWISE_DEQUANTIZED = 0, 1


def quantize_hybrid(x: np.ndarray, fmt_row: int, scale_row, fmt_col: int, scale_col, source: int):
    """Rowwise [rows, cols] codes in fmt_row / scale_row, columnwise [cols, rows] codes in
    fmt_col / scale_col from x (source 0) or from the BF16-dequantized rowwise value (source 1)."""
    assert x.ndim == 2
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    q_row = np.empty((rows, cols), dtype=np.uint8)
    q_col = np.empty((cols, rows), dtype=np.uint8)
    lib().oref_quantize_hybrid(_ptr(x), _dtype_of(x), rows, cols, fmt_row, float(np.float32(scale_row)), fmt_col,
                               float(np.float32(scale_col)), source, _ptr(q_row), _ptr(q_col))
    return q_row, q_col
