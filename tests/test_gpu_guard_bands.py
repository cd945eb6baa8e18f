"""Guard bands: every output of every entry point sits in the middle of a
byte buffer with 64 canary bytes on each side, and the canaries must be
untouched after the call.  Shapes cover full tiles, partial tiles and the
guarded element paths, so an off-by-one in any kernel's edge handling that
writes past its output shows up here (compute-sanitizer is not available).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq

from test_gpu_parity import dev_scalar, random_input

pytestmark = pytest.mark.gpu
E4M3, E5M2 = fq.E4M3, fq.E5M2
PAD = 64
CANARY = 0xA5


class Guarded:
    """Typed views into canary-padded byte buffers, checked together."""

    def __init__(self, dev):
        self.dev, self.bufs = dev, []

    def __call__(self, shape, dtype):
        nbytes = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        buf = torch.full((nbytes + 2 * PAD,), CANARY, dtype=torch.uint8, device=self.dev)
        self.bufs.append((buf, nbytes))
        return buf[PAD:PAD + nbytes].view(dtype).view(shape)

    def check(self):
        torch.cuda.synchronize()
        for i, (buf, nbytes) in enumerate(self.bufs):
            b = buf.cpu().numpy()
            assert np.all(b[:PAD] == CANARY) and np.all(b[PAD + nbytes:] == CANARY), f"output {i} overran"


SHAPES = [(128, 256), (130, 200), (96, 384), (1, 1), (33, 129), (256, 384)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_cast_transpose_and_hybrid(cuda, shape, dtype):
    x = random_input(shape, dtype, 7, cuda)
    r, c = shape
    g = Guarded(cuda)
    q_row, q_col, am = g((r, c), torch.uint8), g((c, r), torch.uint8), g((1,), torch.float32)
    fq.fp8_quantize_cast_transpose(x, E4M3, dev_scalar(0.5, cuda), q_row, q_col, am)
    h_row, h_col = g((r, c), torch.uint8), g((c, r), torch.uint8)
    fq.fp8_quantize_hybrid(x, E4M3, dev_scalar(0.5, cuda), h_row, E5M2, dev_scalar(2.0, cuda), h_col,
                           fq.COLUMNWISE_FROM_ROWWISE_DEQUANTIZED)
    g.check()


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("br", [1, 128])
def test_block_quantize_and_dequantize(cuda, shape, br):
    x = random_input(shape, torch.bfloat16, 8, cuda)
    r, c = shape
    g = Guarded(cuda)
    q, si = g((r, c), torch.uint8), g((-(-r // br), -(-c // 128)), torch.float32)
    fq.fp8_quantize_block(x, br, 128, E4M3, q, si)
    torch.cuda.synchronize()
    y16, y32 = g((r, c), torch.bfloat16), g((r, c), torch.float32)
    fq.fp8_dequantize(q, E4M3, si, y16, br, 128)
    fq.fp8_dequantize(q, E4M3, si, y32, br, 128)
    yt = g((r, c), torch.bfloat16)
    fq.fp8_dequantize(q, E4M3, dev_scalar(1.5, cuda), yt)
    g.check()


@pytest.mark.parametrize("shape", SHAPES + [(100, 70)])
def test_mx(cuda, shape):
    x = random_input(shape, torch.bfloat16, 9, cuda)
    r, c = shape
    g = Guarded(cuda)
    q_row, s_row = g((r, c), torch.uint8), g((r, -(-c // 32)), torch.uint8)
    q_col, s_col = g((c, r), torch.uint8), g((c, -(-r // 32)), torch.uint8)
    fq.fp8_quantize_mx(x, E4M3, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    y = g((r, c), torch.bfloat16)
    fq.fp8_dequantize_mx(q_row, s_row, E4M3, y)
    g.check()


@pytest.mark.parametrize("shape", SHAPES)
def test_block_cast_transpose(cuda, shape):
    x = random_input(shape, torch.bfloat16, 10, cuda)
    r, c = shape
    g = Guarded(cuda)
    q_row, si_row = g((r, c), torch.uint8), g((r, -(-c // 128)), torch.float32)
    q_col, si_col = g((c, r), torch.uint8), g((c, -(-r // 128)), torch.float32)
    fq.fp8_quantize_block_cast_transpose(x, E5M2, q_row, si_row, q_col, si_col)
    g.check()


@pytest.mark.parametrize("n", [1, 17, 4096, 16385, 300_001])
def test_current_delayed_and_grouped(cuda, n):
    x = random_input(n, torch.bfloat16, 11, cuda)
    g = Guarded(cuda)
    q, am, s, si = g((n,), torch.uint8), g((1,), torch.float32), g((1,), torch.float32), g((1,), torch.float32)
    fq.fp8_quantize_current(x, E4M3, q, 0, am, s, si)
    q2, am2, sat = g((n,), torch.uint8), g((1,), torch.float32), g((1,), torch.int64)
    hist = g((7,), torch.float32)
    hist.zero_()
    ds, dsi = g((1,), torch.float32), g((1,), torch.float32)
    ds.fill_(1.0)
    fq.fp8_quantize_delayed(x, E4M3, ds, dsi, q2, hist, 3, fq.AMAX_MAX, 0, am2, sat)
    xs = [x, x[: n // 2 + 1]]
    ga, gs, gsi = g((2,), torch.float32), g((2,), torch.float32), g((2,), torch.float32)
    fq.fp8_amax_grouped(xs, ga, E4M3, 0, gs, gsi)
    qs = [g((t.numel(),), torch.uint8) for t in xs]
    fq.fp8_quantize_grouped(xs, E4M3, gs, qs)
    g.check()
