"""Maximum sizes: tensors of more than 2^31 elements, so that every index on
the device path must be 64-bit.  The oracle (threaded) checks amax, the
saturation count and every code; the dequantized and transposed outputs are
checked on samples against the oracle's per-element rule.

About 13 GB of device memory and 9 GB of host memory.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq

from test_gpu_parity import f32_bits, host_bits

pytestmark = pytest.mark.gpu
E4M3, E5M2 = fq.E4M3, fq.E5M2
N_BIG = (1 << 31) + 33


def big_bf16(shape, seed, dev):
    """BF16 N(0, 1) * 8 filled in slices (no fp32 copy of the whole tensor)."""
    x = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    flat = x.view(-1)
    g = torch.Generator(device=dev).manual_seed(seed)
    step = 1 << 28
    for s in range(0, flat.numel(), step):
        e = min(s + step, flat.numel())
        flat[s:e] = (torch.randn(e - s, generator=g, device=dev) * 8).to(torch.bfloat16)
    return x


def test_amax_quantize_dequantize_beyond_2_pow_31(cuda, oracle):
    threads = oracle.default_threads()
    x = big_bf16((N_BIG,), 71, cuda)
    x[(1 << 31) + 5] = -300.0   # past the 32-bit index range
    x[N_BIG - 1] = 1000.0       # the very last element holds the maximum
    am, s, si = (torch.empty(1, device=cuda) for _ in range(3))
    fq.fp8_amax(x, am, E4M3, 0, s, si)
    torch.cuda.synchronize()
    assert am.item() == 1000.0
    xb = host_bits(x)
    ws, wsi = oracle.compute_scale(np.float32(1000.0), E4M3, 0)
    assert (f32_bits(s.item()), f32_bits(si.item())) == (f32_bits(ws), f32_bits(wsi))
    # a scale that saturates everything above 100: the count covers the whole range
    scale = torch.full((1,), 4.48, device=cuda)
    q = torch.empty(N_BIG, dtype=torch.uint8, device=cuda)
    am2 = torch.empty(1, device=cuda)
    sat = torch.empty(1, dtype=torch.int64, device=cuda)
    fq.fp8_quantize(x, E4M3, scale, q, am2, sat)
    torch.cuda.synchronize()
    wq, wsat = oracle.quantize(xb, E4M3, np.float32(4.48), threads)
    assert sat.item() == wsat and wsat >= 2
    assert am2.item() == 1000.0
    assert np.array_equal(q.cpu().numpy(), wq)
    del wq
    y = torch.empty(N_BIG, dtype=torch.bfloat16, device=cuda)
    si2 = torch.full((1,), np.float32(1.0) / np.float32(4.48), device=cuda)
    fq.fp8_dequantize(q, E4M3, si2, y)
    torch.cuda.synchronize()
    idx = torch.cat([torch.randint(0, N_BIG, (1 << 20,), device=cuda),
                     torch.arange(N_BIG - 4096, N_BIG, device=cuda)])
    qs = q[idx].cpu().numpy()
    want = oracle.dequantize(qs, E4M3, si2.cpu().numpy())
    assert np.array_equal(host_bits(y[idx]), want)


def test_cast_transpose_beyond_2_pow_31(cuda, oracle):
    rows, cols = 16512, 131072  # 2.16e9 elements, 129 x 1024 tiles
    x = big_bf16((rows, cols), 72, cuda)
    x[rows - 1, cols - 1] = 512.0
    scale = torch.full((1,), 0.5, device=cuda)
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    am = torch.empty(1, device=cuda)
    # 132096 tiles: the fused amax walks them with 8192 CTAs
    fq.fp8_quantize_cast_transpose(x, E4M3, scale, q_row, None, am)
    fq.fp8_quantize_cast_transpose(x, E4M3, scale, None, q_col)
    torch.cuda.synchronize()
    assert am.item() == 512.0
    g = torch.Generator(device=cuda).manual_seed(3)
    r = torch.cat([torch.randint(0, rows, (1 << 20,), generator=g, device=cuda),
                   torch.full((256,), rows - 1, device=cuda)])
    c = torch.cat([torch.randint(0, cols, (1 << 20,), generator=g, device=cuda),
                   torch.arange(cols - 256, cols, device=cuda)])
    wq, _ = oracle.quantize(host_bits(x[r, c]), E4M3, np.float32(0.5))
    assert np.array_equal(q_row[r, c].cpu().numpy(), wq)
    assert np.array_equal(q_col[c, r].cpu().numpy(), wq)


def test_blockwise_beyond_2_pow_31(cuda, oracle):
    """128 x 128 and 1 x 128 block scaling, and the 1 x 128 blockwise dequantize,
    on 16512 x 131072 BF16; the last 256 rows (offsets past 2^31) are checked
    code by code and scale by scale against the oracle."""
    rows, cols = 16512, 131072
    x = big_bf16((rows, cols), 73, cuda)
    tail = slice(rows - 256, rows)
    xt = host_bits(x[tail])
    for br in (128, 1):
        q = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
        si = torch.empty((-(-rows // br), cols // 128), dtype=torch.float32, device=cuda)
        fq.fp8_quantize_block(x, br, 128, E4M3, q, si)
        torch.cuda.synchronize()
        wq, wsi = oracle.quantize_block(xt, br, 128, E4M3, oracle.default_threads())
        assert np.array_equal(q[tail].cpu().numpy(), wq), br
        sit = si[(rows - 256) // br:] if br == 128 else si[tail]
        assert np.array_equal(sit.cpu().numpy().view(np.uint32), wsi.view(np.uint32)), br
        if br == 1:
            y = torch.empty((rows, cols), dtype=torch.bfloat16, device=cuda)
            fq.fp8_dequantize(q, E4M3, si, y, 1, 128)
            torch.cuda.synchronize()
            wy = oracle.dequantize(wq, E4M3, wsi, 1, 128, threads=oracle.default_threads())
            assert np.array_equal(host_bits(y[tail]), wy)
            del y
        del q, si


def test_tall_tensors_past_65535_row_tiles(cuda, oracle):
    """Shapes with more than 65535 rows of tiles (the kernels index tiles
    linearly): MXFP8, 128 x 128 blocks and the blockwise cast-transpose (all
    128-row tiles); the last rows against the oracle."""
    rows = 65536 * 128 + 160  # 65538 rows of MX tiles, the last one 32 rows high
    x = big_bf16((rows, 128), 74, cuda)
    q = torch.empty((rows, 128), dtype=torch.uint8, device=cuda)
    s = torch.empty((rows, 4), dtype=torch.uint8, device=cuda)
    qc = torch.empty((128, rows), dtype=torch.uint8, device=cuda)
    sc = torch.empty((128, rows // 32), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_mx(x, E4M3, q, s, qc, sc)
    torch.cuda.synchronize()
    tail = host_bits(x[-256:])
    wq, ws = oracle.quantize_mx(tail, E4M3)
    assert np.array_equal(q[-256:].cpu().numpy(), wq) and np.array_equal(s[-256:].cpu().numpy(), ws)
    wq, ws = oracle.quantize_mx(np.ascontiguousarray(tail.T), E4M3)
    assert np.array_equal(qc[:, -256:].cpu().numpy(), wq) and np.array_equal(sc[:, -8:].cpu().numpy(), ws)
    del x, q, s, qc, sc
    rows = 65536 * 128 + 256  # 8,388,864 rows: 65538 row blocks of 128
    x = big_bf16((rows, 128), 75, cuda)
    tail = host_bits(x[-256:])
    q = torch.empty((rows, 128), dtype=torch.uint8, device=cuda)
    si = torch.empty((rows // 128, 1), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block(x, 128, 128, E4M3, q, si)
    torch.cuda.synchronize()
    wq, wsi = oracle.quantize_block(tail, 128, 128, E4M3)
    assert np.array_equal(q[-256:].cpu().numpy(), wq) and np.array_equal(si[-2:].cpu().numpy(), wsi)
    q_row = torch.empty((rows, 128), dtype=torch.uint8, device=cuda)
    s_row = torch.empty((rows, 1), dtype=torch.float32, device=cuda)
    q_col = torch.empty((128, rows), dtype=torch.uint8, device=cuda)
    s_col = torch.empty((128, rows // 128), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block_cast_transpose(x, E4M3, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    wq, wsi = oracle.quantize_block(tail, 1, 128, E4M3)
    assert np.array_equal(q_row[-256:].cpu().numpy(), wq) and np.array_equal(s_row[-256:].cpu().numpy(), wsi)
    wqt, wst = oracle.quantize_block(np.ascontiguousarray(tail.T), 1, 128, E4M3)
    assert np.array_equal(q_col[:, -256:].cpu().numpy(), wqt)
    assert np.array_equal(s_col[:, -2:].cpu().numpy(), wst)
