"""Every BF16 magnitude as a block amax: the block scale rule, exhaustively.

"Low Precision Training and Rollout" (FP32 scale per 128 x 128 block, the
stored factor the inverse scale) with the per-tensor rule of "Megatron FP8"
§4 (scale = FP8_MAX / amax, scale_inv = 1 / scale, margin 0).  The BF16 block
kernels derive scale and scale_inv of BF16 data from exact tables instead of
two divisions; the rule has one input, the amax, and a BF16 amax has 32768
possible bit patterns (sign cleared).  Each test gives every pattern -- zero,
subnormals, normals, Inf and every NaN -- to a 1 x 128 row tile or a 128 x 1
column tile (both directions of the blockwise cast-transpose), and a spread
of them to 128 x 128 blocks, and compares scale_inv and every code with the
oracle bit for bit, for both formats.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq

pytestmark = pytest.mark.gpu
FMTS = [fq.E4M3, fq.E5M2]


def rows_with_maxima(patterns: np.ndarray, width: int, seed: int) -> np.ndarray:
    """uint16 BF16 bits [len(patterns), width]: row r holds the magnitude
    patterns[r] once (random sign, random column) and elsewhere random
    magnitudes not above it (random signs), so the row's amax is patterns[r]."""
    rng = np.random.default_rng(seed)
    n = len(patterns)
    p = patterns.astype(np.uint32)[:, None]
    mags = (rng.integers(0, 1 << 16, size=(n, width), dtype=np.uint32) * (p + 1)) >> 16  # in [0, p]
    col = rng.integers(0, width, size=n)
    mags[np.arange(n), col] = patterns
    signs = rng.integers(0, 2, size=(n, width), dtype=np.uint32) << 15
    return (mags | signs).astype(np.uint16)


def to_device(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)


ALL = np.arange(0x8000, dtype=np.uint16)  # every non-negative BF16 bit pattern


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bf16_amax_in_1x128_tiles(cuda, oracle, fmt):
    xb = rows_with_maxima(ALL, 128, 1 + fmt)
    x = to_device(xb, cuda)
    q = torch.empty(xb.shape, dtype=torch.uint8, device=cuda)
    si = torch.empty((xb.shape[0], 1), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block(x, 1, 128, fmt, q, si)
    torch.cuda.synchronize()
    wq, wsi = oracle.quantize_block(xb, 1, 128, fmt)
    assert np.array_equal(si.cpu().numpy().view(np.uint32), wsi.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), wq)


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bf16_amax_in_block_cast_transpose(cuda, oracle, fmt):
    """Rowwise: [32768, 128], one row tile per pattern.  Columnwise: the
    transpose, [128, 32768], one column tile per pattern."""
    xb = rows_with_maxima(ALL, 128, 3 + fmt)
    for bits in (xb, np.ascontiguousarray(xb.T)):
        rows, cols = bits.shape
        x = to_device(bits, cuda)
        q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
        s_row = torch.empty((rows, cols // 128), dtype=torch.float32, device=cuda)
        q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
        s_col = torch.empty((cols, rows // 128), dtype=torch.float32, device=cuda)
        fq.fp8_quantize_block_cast_transpose(x, fmt, q_row, s_row, q_col, s_col)
        torch.cuda.synchronize()
        wq, ws = oracle.quantize_block(bits, 1, 128, fmt)
        assert np.array_equal(s_row.cpu().numpy().view(np.uint32), ws.view(np.uint32))
        assert np.array_equal(q_row.cpu().numpy(), wq)
        wqt, wst = oracle.quantize_block(np.ascontiguousarray(bits.T), 1, 128, fmt)
        assert np.array_equal(s_col.cpu().numpy().view(np.uint32), wst.view(np.uint32))
        assert np.array_equal(q_col.cpu().numpy(), wqt)


@pytest.mark.parametrize("fmt", FMTS)
def test_bf16_amax_spread_in_128x128_blocks(cuda, oracle, fmt):
    """1024 patterns (every 32nd, plus the exponent edges, Inf and NaN) as the
    maxima of 128 x 128 blocks: x is [128, 128 * 1024]."""
    pats = np.unique(np.concatenate([ALL[::32], np.array([0, 1, 0x7F, 0x80, 0x3F80, 0x3FFF, 0x7F7F, 0x7F80,
                                                          0x7F81, 0x7FC0, 0x7FFF, 0x0080, 0x00FF], np.uint16)]))
    pats = np.concatenate([pats, ALL[1::97]])[:1024]
    blocks = rows_with_maxima(pats, 128 * 128, 13 + fmt).reshape(len(pats), 128, 128)
    xb = np.ascontiguousarray(blocks.transpose(1, 0, 2).reshape(128, len(pats) * 128))
    x = to_device(xb, cuda)
    q = torch.empty(xb.shape, dtype=torch.uint8, device=cuda)
    si = torch.empty((1, len(pats)), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block(x, 128, 128, fmt, q, si)
    torch.cuda.synchronize()
    wq, wsi = oracle.quantize_block(xb, 128, 128, fmt)
    assert np.array_equal(si.cpu().numpy().view(np.uint32), wsi.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), wq)
