"""GB300-native FP8 scaled quantization.

Python binding of the C ABI in ``include/fp8q.h``.  Every function here only
marshals arguments (tensor data pointers, sizes, the current CUDA stream) and
calls the CUDA library; all arithmetic runs in the library's sm_103a kernels.
Tensors must be contiguous CUDA tensors; BF16 / fp32 inputs, uint8 codes,
fp32 scalars, int64 saturation counters (read as unsigned 64-bit).

Entry points (same names as the C ABI):
  fp8_amax, fp8_update_scale_delayed, fp8_quantize,
  fp8_quantize_cast_transpose, fp8_quantize_block, fp8_dequantize.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

E4M3, E5M2 = 0, 1
DT_BF16, DT_FP32 = 0, 1
AMAX_MAX, AMAX_MOST_RECENT = 0, 1
COLUMNWISE_FROM_ORIGINAL, COLUMNWISE_FROM_ROWWISE_DEQUANTIZED = 0, 1
FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}

__all__ = [
    "E4M3", "E5M2", "DT_BF16", "DT_FP32", "AMAX_MAX", "AMAX_MOST_RECENT", "FP8_MAX", "Fp8Error",
    "fp8_amax", "fp8_update_scale_delayed", "fp8_quantize", "fp8_quantize_cast_transpose",
    "fp8_quantize_block", "fp8_dequantize", "fp8_quantize_delayed", "fp8_quantize_mx", "fp8_dequantize_mx",
    "fp8_block128_scales_to_mx", "fp8_amax_noalloc", "fp8_quantize_current", "fp8_quantize_hybrid", "fp8_quantize_block_cast_transpose",
    "fp8_amax_grouped", "fp8_quantize_grouped", "COLUMNWISE_FROM_ORIGINAL", "COLUMNWISE_FROM_ROWWISE_DEQUANTIZED",
    "launch_count", "version", "library", "release_stream_workspace", "wait_timeouts",
]


class Fp8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} [status {status}]")
        self.status = status


def library():
    """The loaded ctypes library (raises if it has not been built)."""
    return _lib.load()


def version() -> int:
    return library().fp8_version()


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(library().fp8_launch_count())


def wait_timeouts() -> int:
    """Waits inside the library's tile pipelines that gave up on the current
    device since the library was loaded (synchronises the device).  Any change
    across a call means that call's outputs are incomplete."""
    import ctypes
    count = ctypes.c_ulonglong(0)
    _check(library().fp8_wait_timeouts(ctypes.addressof(count)))
    return int(count.value)


def release_stream_workspace(stream=None):
    """Free the library's reduction workspace of `stream` (default: the current
    stream) on the current device, after the stream's queued work."""
    _check(library().fp8_release_stream_workspace(_stream(stream)))


def _check(status: int):
    if status != 0:
        msg = library().fp8_last_error_message().decode(errors="replace")
        raise Fp8Error(status, msg)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DT_BF16
    if t.dtype == torch.float32:
        return DT_FP32
    raise TypeError(f"expected a bfloat16 or float32 tensor, got {t.dtype}")


def _p(t) -> int | None:
    """Data pointer of an optional contiguous tensor on the current CUDA device
    (the library launches on the current device's stream, so a tensor on
    another device would be reached through a peer pointer)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a tensor, got {type(t)}")
    if not t.is_cuda:
        raise ValueError("tensors passed to the FP8 library must live on a CUDA device")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device}, but the current CUDA device is cuda:{torch.cuda.current_device()}; "
                         "call inside `with torch.cuda.device(...)`")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the FP8 library must be contiguous")
    return t.data_ptr() or None


def _f32(t, name: str) -> int | None:
    """Pointer of an optional fp32 device scalar (amax, scale, scale_inv): the
    library reads or writes one 4-byte word there."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.numel() < 1:
        raise ValueError(f"{name} must be a float32 tensor of at least one element")
    return _p(t)


def _u64(t, name: str) -> int | None:
    """Pointer of an optional 64-bit device counter (the saturation count)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype not in (torch.int64, torch.uint64) or t.numel() < 1:
        raise ValueError(f"{name} must be an int64 tensor of at least one element")
    return _p(t)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _rows_cols(x: torch.Tensor):
    if x.dim() != 2:
        raise ValueError(f"expected a 2-D tensor, got shape {tuple(x.shape)}")
    return int(x.shape[0]), int(x.shape[1])


def fp8_amax(x, amax_out, fmt=E4M3, margin=0, scale_out=None, scale_inv_out=None, stream=None):
    """amax_out[0] = max|x|; with scale_out / scale_inv_out, also the current scale."""
    _check(library().fp8_amax(_p(x), _dt(x), x.numel(), _f32(amax_out, "amax_out"), fmt, margin,
                              _f32(scale_out, "scale_out"), _f32(scale_inv_out, "scale_inv_out"), _stream(stream)))


def fp8_quantize_mx(x, fmt, q_row=None, scale_row=None, q_col=None, scale_col=None, stream=None):
    """MXFP8: codes with one E8M0 scale per 32 elements, rowwise ([rows, cols] codes,
    [rows, ceil(cols/32)] scales) and/or columnwise (transposed: [cols, rows] codes,
    [cols, ceil(rows/32)] scales)."""
    rows, cols = _rows_cols(x)
    for t, shape in ((q_row, (rows, cols)), (scale_row, (rows, -(-cols // 32))), (q_col, (cols, rows)),
                     (scale_col, (cols, -(-rows // 32)))):
        if t is not None and (t.dtype != torch.uint8 or tuple(t.shape) != shape):
            raise ValueError(f"MX outputs must be uint8 {shape}")
    _check(library().fp8_quantize_mx(_p(x), _dt(x), rows, cols, fmt, _p(q_row), _p(scale_row), _p(q_col),
                                     _p(scale_col), _stream(stream)))


def fp8_dequantize_mx(q, scales, fmt, y, stream=None):
    """y = decode(q) * 2^(scale - 127) for rowwise MX data [rows, cols]."""
    rows, cols = _rows_cols(q)
    if scales.dtype != torch.uint8 or tuple(scales.shape) != (rows, -(-cols // 32)):
        raise ValueError("scales must be uint8 [rows, ceil(cols/32)]")
    if tuple(y.shape) != (rows, cols):
        raise ValueError("y must have q's shape")
    _check(library().fp8_dequantize_mx(_p(q), _p(scales), fmt, rows, cols, _p(y), _dt(y), _stream(stream)))


def fp8_block128_scales_to_mx(scale_inv, rows, cols, mx_scales, bad_blocks_out=None, stream=None):
    """E8M0 1x32 scales from power-of-two 128x128 block scale_inv (codes unchanged)."""
    if scale_inv.dtype != torch.float32 or mx_scales.dtype != torch.uint8:
        raise TypeError("scale_inv must be float32 and mx_scales uint8")
    if tuple(mx_scales.shape) != (rows, -(-cols // 32)):
        raise ValueError("mx_scales must be uint8 [rows, ceil(cols/32)]")
    _check(library().fp8_block128_scales_to_mx(_p(scale_inv), rows, cols, _p(mx_scales),
                                               _u64(bad_blocks_out, "bad_blocks_out"), _stream(stream)))


def fp8_amax_noalloc(x, amax_out, fmt=E4M3, margin=0, scale_out=None, scale_inv_out=None, stream=None):
    """fp8_amax for callers that cannot allocate device memory: the library
    uses a fixed file-scope scratch array instead of a per-stream workspace.
    At most 2**28 elements; make the first call on a device before any stream
    capture; calls that overlap on the GPU race on the shared scratch."""
    _check(library().fp8_amax_noalloc(_p(x), _dt(x), x.numel(), _f32(amax_out, "amax_out"), fmt, margin,
                                      _f32(scale_out, "scale_out"), _f32(scale_inv_out, "scale_inv_out"),
                                      _stream(stream)))


def fp8_update_scale_delayed(amax_history, step, new_amax, algo, fmt, margin, scale_out, scale_inv_out,
                             stream=None):
    """Delayed-scaling update of a float32 history (in place) -> scale_out, scale_inv_out."""
    if amax_history.dtype != torch.float32:
        raise TypeError("amax_history must be float32")
    _check(library().fp8_update_scale_delayed(_p(amax_history), amax_history.numel(), int(step),
                                              _f32(new_amax, "new_amax"), algo, fmt, margin,
                                              _f32(scale_out, "scale_out"), _f32(scale_inv_out, "scale_inv_out"),
                                              _stream(stream)))


def fp8_quantize(x, fmt, scale, q_out, amax_out=None, sat_count_out=None, stream=None):
    """q_out = FP8 codes of x * scale; optional fused amax and saturation count."""
    if q_out.dtype != torch.uint8:
        raise TypeError("q_out must be uint8")
    if q_out.numel() != x.numel():
        raise ValueError("q_out must have as many elements as x")
    _check(library().fp8_quantize(_p(x), _dt(x), x.numel(), fmt, _f32(scale, "scale"), _p(q_out),
                                  _f32(amax_out, "amax_out"), _u64(sat_count_out, "sat_count_out"),
                                  _stream(stream)))


def fp8_quantize_delayed(x, fmt, scale, scale_inv, q_out, amax_history, step, algo=AMAX_MAX, margin=0,
                         amax_out=None, sat_count_out=None, stream=None):
    """One delayed-scaling step in one call (the cast, then a one-CTA finalize):
    q_out = codes of x * scale, then
    amax(x) goes into amax_history[step % len] and scale / scale_inv are
    overwritten with the scale of the next step."""
    if q_out.dtype != torch.uint8 or q_out.numel() != x.numel():
        raise ValueError("q_out must be uint8 with as many elements as x")
    if amax_history.dtype != torch.float32:
        raise TypeError("amax_history must be float32")
    _check(library().fp8_quantize_delayed(_p(x), _dt(x), x.numel(), fmt, _f32(scale, "scale"),
                                          _f32(scale_inv, "scale_inv"), _p(q_out), _p(amax_history),
                                          amax_history.numel(), int(step), algo, margin, _f32(amax_out, "amax_out"),
                                          _u64(sat_count_out, "sat_count_out"), _stream(stream)))


def fp8_quantize_cast_transpose(x, fmt, scale, q_row, q_col, amax_out=None, stream=None):
    """Rowwise [rows, cols] and columnwise [cols, rows] codes under one scale."""
    rows, cols = _rows_cols(x)
    if q_row is not None and (q_row.dtype != torch.uint8 or tuple(q_row.shape) != (rows, cols)):
        raise ValueError("q_row must be uint8 [rows, cols]")
    if q_col is not None and (q_col.dtype != torch.uint8 or tuple(q_col.shape) != (cols, rows)):
        raise ValueError("q_col must be uint8 [cols, rows]")
    _check(library().fp8_quantize_cast_transpose(_p(x), _dt(x), rows, cols, fmt, _f32(scale, "scale"), _p(q_row),
                                                 _p(q_col), _f32(amax_out, "amax_out"), _stream(stream)))


def fp8_quantize_block(x, block_rows, block_cols, fmt, q_out, scale_inv_out, stream=None):
    """Block-scaled codes and per-block scale_inv ([ceil(r/br), ceil(c/bc)] fp32)."""
    rows, cols = _rows_cols(x)
    if q_out.dtype != torch.uint8 or tuple(q_out.shape) != (rows, cols):
        raise ValueError("q_out must be uint8 [rows, cols]")
    if block_rows > 0 and block_cols > 0:
        want = (-(-rows // block_rows), -(-cols // block_cols))
        if scale_inv_out.dtype != torch.float32 or tuple(scale_inv_out.shape) != want:
            raise ValueError(f"scale_inv_out must be float32 {want}")
    _check(library().fp8_quantize_block(_p(x), _dt(x), rows, cols, block_rows, block_cols, fmt, _p(q_out),
                                        _p(scale_inv_out), _stream(stream)))


def fp8_dequantize(q, fmt, scale_inv, y, block_rows=0, block_cols=0, stream=None):
    """y = decode(q) * scale_inv (fp32 multiply) stored as y's dtype (bf16 / fp32)."""
    if q.dtype != torch.uint8:
        raise TypeError("q must be uint8")
    if y.numel() != q.numel():
        raise ValueError("y must have as many elements as q")
    if q.dim() == 2:
        rows, cols = int(q.shape[0]), int(q.shape[1])
    else:
        if block_rows or block_cols:
            raise ValueError("block-scaled dequantize needs a 2-D q")
        rows, cols = 1, q.numel()
    if block_rows > 0 and block_cols > 0:
        nblocks = -(-rows // block_rows) * -(-cols // block_cols)
        if scale_inv.dtype != torch.float32 or scale_inv.numel() < nblocks:
            raise ValueError(f"block scale_inv must be float32 with at least {nblocks} elements")
        si = _p(scale_inv)
    else:
        si = _f32(scale_inv, "scale_inv")
    _check(library().fp8_dequantize(_p(q), fmt, rows, cols, si, block_rows, block_cols, _p(y),
                                    _dt(y), _stream(stream)))


def fp8_quantize_hybrid(x, fmt_row, scale_row, q_row, fmt_col, scale_col, q_col,
                        source=COLUMNWISE_FROM_ORIGINAL, stream=None):
    """Rowwise codes (fmt_row, scale_row) and transposed columnwise codes (fmt_col,
    scale_col) from x or from the BF16-dequantized rowwise value."""
    rows, cols = _rows_cols(x)
    if q_row.dtype != torch.uint8 or tuple(q_row.shape) != (rows, cols):
        raise ValueError("q_row must be uint8 [rows, cols]")
    if q_col.dtype != torch.uint8 or tuple(q_col.shape) != (cols, rows):
        raise ValueError("q_col must be uint8 [cols, rows]")
    _check(library().fp8_quantize_hybrid(_p(x), _dt(x), rows, cols, fmt_row, _f32(scale_row, "scale_row"),
                                         _p(q_row), fmt_col, _f32(scale_col, "scale_col"), _p(q_col), source,
                                         _stream(stream)))


def fp8_quantize_block_cast_transpose(x, fmt, q_row=None, scale_inv_row=None, q_col=None, scale_inv_col=None,
                                      stream=None):
    """1 x 128 blockwise codes of x ([rows, cols] + fp32 [rows, ceil(cols/128)]) and of
    x^T ([cols, rows] + fp32 [cols, ceil(rows/128)]) from one read of x."""
    rows, cols = _rows_cols(x)
    for t, shape, dt in ((q_row, (rows, cols), torch.uint8), (scale_inv_row, (rows, -(-cols // 128)), torch.float32),
                         (q_col, (cols, rows), torch.uint8), (scale_inv_col, (cols, -(-rows // 128)), torch.float32)):
        if t is not None and (t.dtype != dt or tuple(t.shape) != shape):
            raise ValueError(f"block cast-transpose outputs must be {dt} {shape}")
    _check(library().fp8_quantize_block_cast_transpose(_p(x), _dt(x), rows, cols, fmt, _p(q_row), _p(scale_inv_row),
                                                       _p(q_col), _p(scale_inv_col), _stream(stream)))


def _ptr_array(tensors):
    return (ctypes.c_void_p * len(tensors))(*[_p(t) for t in tensors])


def fp8_amax_grouped(xs, amax_out=None, fmt=E4M3, margin=0, scale_out=None, scale_inv_out=None, stream=None):
    """Per-tensor amax (and current scale) of up to 128 tensors in one launch (+ finalize);
    outputs are float32 device tensors of at least len(xs) elements."""
    if not xs or len({t.dtype for t in xs}) != 1:
        raise ValueError("xs must be a non-empty list of tensors of one dtype")
    for out in (amax_out, scale_out, scale_inv_out):
        if out is not None and (out.dtype != torch.float32 or out.numel() < len(xs)):
            raise ValueError("grouped outputs must be float32 tensors of at least len(xs) elements")
    ns = (ctypes.c_int64 * len(xs))(*[t.numel() for t in xs])
    _check(library().fp8_amax_grouped(len(xs), _ptr_array(xs), ns, _dt(xs[0]), _p(amax_out), fmt, margin,
                                      _p(scale_out), _p(scale_inv_out), _stream(stream)))


def fp8_quantize_grouped(xs, fmt, scales, qs, stream=None):
    """qs[i] = codes of xs[i] * scales[i] for up to 128 tensors in one kernel launch."""
    if not xs or len(xs) != len(qs) or len({t.dtype for t in xs}) != 1:
        raise ValueError("xs and qs must be equally long lists; xs of one dtype")
    for x, q in zip(xs, qs):
        if q.dtype != torch.uint8 or q.numel() != x.numel():
            raise ValueError("each q must be uint8 with as many elements as its x")
    if scales.dtype != torch.float32 or scales.numel() < len(xs):
        raise ValueError("scales must be a float32 tensor of at least len(xs) elements")
    ns = (ctypes.c_int64 * len(xs))(*[t.numel() for t in xs])
    _check(library().fp8_quantize_grouped(len(xs), _ptr_array(xs), ns, _dt(xs[0]), fmt, _p(scales), _ptr_array(qs),
                                          _stream(stream)))


def fp8_quantize_current(x, fmt, q_out, margin=0, amax_out=None, scale_out=None, scale_inv_out=None, stream=None):
    """Current scaling in one call: amax(x), the scale with `margin`, and q_out = codes
    of x * scale (the cast reduces the amax partials itself; no separate finalize)."""
    if q_out.dtype != torch.uint8:
        raise TypeError("q_out must be uint8")
    if q_out.numel() != x.numel():
        raise ValueError("q_out must have as many elements as x")
    _check(library().fp8_quantize_current(_p(x), _dt(x), x.numel(), fmt, margin, _p(q_out),
                                          _f32(amax_out, "amax_out"), _f32(scale_out, "scale_out"),
                                          _f32(scale_inv_out, "scale_inv_out"), _stream(stream)))
