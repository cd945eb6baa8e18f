"""GPU parity of the MXFP8 entry points against the oracle (bit for bit):
rowwise / columnwise E8M0-scaled codes, MX dequantize, and the lossless
128x128 -> 1x32 scale re-blocking."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq
from fp8_scaled_quantization_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

E4M3, E5M2 = fq.E4M3, fq.E5M2


def host(x):
    h = x.detach().contiguous().cpu()
    return h.view(torch.int16).numpy().view(np.uint16) if h.dtype == torch.bfloat16 else h.numpy()


def mx_input(shape, dtype, seed, dev, specials=True):
    g = torch.Generator(device="cpu").manual_seed(seed)
    rows, cols = shape
    mags = torch.exp(3 * torch.randn((rows, max(1, -(-cols // 32))), generator=g))
    mags = mags.repeat_interleave(32, 1)[:, :cols]
    x = torch.randn(shape, generator=g) * mags
    if specials and x.numel() > 200:
        flat = x.view(-1)
        flat[7] = float("inf")
        flat[100] = float("nan")
        flat[150:182] = 0.0
        flat[-1] = 1e-39
    return x.to(dtype).to(dev)


# 32-row multiples with 128-column multiples take the 128 x 128-tile kernel
# (its last row of tiles 32, 64, 96 or 128 rows high), the rest the guarded
# kernel.
SHAPES = [(32, 128), (64, 384), (96, 256), (33, 130), (1, 31), (100, 64), (7, 1000), (256, 4096), (128, 128),
          (384, 256), (160, 256), (224, 128)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", SHAPES)
def test_mx_quantize_matches_oracle(cuda, oracle, dtype, fmt, shape):
    rows, cols = shape
    x = mx_input(shape, dtype, rows * 31 + cols, cuda)
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    s_row = torch.empty((rows, -(-cols // 32)), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    s_col = torch.empty((cols, -(-rows // 32)), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_mx(x, fmt, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    xb = host(x)
    wq, ws = oracle.quantize_mx(xb, fmt)
    assert np.array_equal(s_row.cpu().numpy(), ws)
    assert np.array_equal(q_row.cpu().numpy(), wq)
    wqt, wst = oracle.quantize_mx(np.ascontiguousarray(xb.T), fmt)
    assert np.array_equal(s_col.cpu().numpy(), wst)
    assert np.array_equal(q_col.cpu().numpy(), wqt)


def test_mx_signed_special_blocks(cuda, oracle):
    """Blocks of -0.0, all-subnormal blocks of both signs, -Inf among normals,
    negative NaNs and +-BF16 max with equal magnitudes, in both directions of
    the 128 x 128-tile kernel."""
    x = mx_input((64, 256), torch.float32, 17, "cpu", specials=False)
    v = x.view(-1)
    v[0:32] = -0.0
    sub = torch.tensor([1e-39, -2e-39, 5e-40, -9e-41], dtype=torch.float32)
    v[32:64] = sub.repeat(8)
    v[64 + 5] = float("-inf")
    v[96 + 3] = -float("nan")
    v[128:160] = torch.tensor([3.3895e38, -3.3895e38] * 16)
    v[160:192] = torch.tensor([-2.0, 2.0] * 16)
    x[:, 200] = -0.0          # a column of -0.0 (columnwise blocks)
    x[0:32, 201] = -1e-39     # a columnwise all-subnormal block
    x[40, 202] = float("-inf")
    x = x.to(torch.bfloat16).to(cuda)
    rows, cols = x.shape
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    s_row = torch.empty((rows, cols // 32), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    s_col = torch.empty((cols, rows // 32), dtype=torch.uint8, device=cuda)
    for fmt in (E4M3, E5M2):
        fq.fp8_quantize_mx(x, fmt, q_row, s_row, q_col, s_col)
        torch.cuda.synchronize()
        xb = host(x)
        wq, ws = oracle.quantize_mx(xb, fmt)
        assert np.array_equal(s_row.cpu().numpy(), ws) and np.array_equal(q_row.cpu().numpy(), wq)
        wqt, wst = oracle.quantize_mx(np.ascontiguousarray(xb.T), fmt)
        assert np.array_equal(s_col.cpu().numpy(), wst) and np.array_equal(q_col.cpu().numpy(), wqt)


def test_mx_single_direction(cuda, oracle):
    x = mx_input((64, 256), torch.bfloat16, 5, cuda)
    q = torch.empty((256, 64), dtype=torch.uint8, device=cuda)
    s = torch.empty((256, 2), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_mx(x, E4M3, None, None, q, s)
    torch.cuda.synchronize()
    wq, ws = oracle.quantize_mx(np.ascontiguousarray(host(x).T), E4M3)
    assert np.array_equal(q.cpu().numpy(), wq) and np.array_equal(s.cpu().numpy(), ws)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", [(37, 100), (64, 256), (3, 4096), (1, 32)])
def test_mx_dequantize_matches_oracle(cuda, oracle, out_dtype, fmt, shape):
    # (37, 100): the general kernel; the others have cols % 32 == 0 (vector kernel)
    rows, cols = shape
    g = torch.Generator(device="cpu").manual_seed(3 + rows)
    q = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
    s = torch.randint(0, 256, (rows, -(-cols // 32)), generator=g, dtype=torch.uint8)
    s.view(-1)[:4] = torch.tensor([0, 1, 254, 255], dtype=torch.uint8)[: s.numel()]
    y = torch.empty(shape, dtype=out_dtype, device=cuda)
    fq.fp8_dequantize_mx(q.to(cuda), s.to(cuda), fmt, y)
    torch.cuda.synchronize()
    want = oracle.dequantize_mx(q.numpy(), s.numpy(), fmt, out_dt=oracle.BF16 if out_dtype == torch.bfloat16 else oracle.FP32)
    got = host(y)
    assert np.array_equal(got.view(np.uint32) if out_dtype == torch.float32 else got,
                          want.view(np.uint32) if out_dtype == torch.float32 else want)


def test_block128_to_mx_rescale_matches_oracle(cuda, oracle):
    rows, cols = 300, 520
    g = torch.Generator(device="cpu").manual_seed(9)
    k = torch.randint(-140, 128, (3, 5), generator=g)
    si = torch.pow(2.0, k.double()).float()
    si[1, 1] = 3.0       # not a power of two
    si[2, 4] = 2.0 ** -130  # below the E8M0 range
    out = torch.empty((rows, -(-cols // 32)), dtype=torch.uint8, device=cuda)
    bad = torch.empty(1, dtype=torch.int64, device=cuda)
    fq.fp8_block128_scales_to_mx(si.to(cuda), rows, cols, out, bad)
    torch.cuda.synchronize()
    want, wbad = oracle.block128_scales_to_mx(si.numpy(), rows, cols)
    assert np.array_equal(out.cpu().numpy(), want)
    assert bad.item() == wbad >= 2


def test_block128_to_mx_empty_shape_clears_the_count(cuda):
    bad = torch.full((1,), 7, dtype=torch.int64, device=cuda)
    out = torch.empty((0, 4), dtype=torch.uint8, device=cuda)
    fq.fp8_block128_scales_to_mx(torch.empty((0, 1), device=cuda), 0, 128, out, bad)
    torch.cuda.synchronize()
    assert bad.item() == 0


def test_mx_full_size_activation(cuda, oracle):
    x = wl.w2_student_t(device=cuda)  # 8192 x 8192 BF16
    rows, cols = x.shape
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    s_row = torch.empty((rows, cols // 32), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    s_col = torch.empty((cols, rows // 32), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_mx(x, E4M3, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    xb = host(x)
    th = oracle.default_threads()
    wq, ws = oracle.quantize_mx(xb, E4M3, th)
    assert np.array_equal(s_row.cpu().numpy(), ws) and np.array_equal(q_row.cpu().numpy(), wq)
    del wq
    wqt, wst = oracle.quantize_mx(np.ascontiguousarray(xb.T), E4M3, th)
    assert np.array_equal(s_col.cpu().numpy(), wst) and np.array_equal(q_col.cpu().numpy(), wqt)


@pytest.mark.parametrize("which", ["rowwise", "columnwise"])
def test_mx_single_direction_several_tiles(cuda, oracle, which):
    x = mx_input((256, 384), torch.bfloat16, 6, cuda)
    if which == "rowwise":
        q = torch.empty((256, 384), dtype=torch.uint8, device=cuda)
        s = torch.empty((256, 12), dtype=torch.uint8, device=cuda)
        fq.fp8_quantize_mx(x, E5M2, q, s)
        want = oracle.quantize_mx(host(x), E5M2)
    else:
        q = torch.empty((384, 256), dtype=torch.uint8, device=cuda)
        s = torch.empty((384, 8), dtype=torch.uint8, device=cuda)
        fq.fp8_quantize_mx(x, E5M2, None, None, q, s)
        want = oracle.quantize_mx(np.ascontiguousarray(host(x).T), E5M2)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), want[0]) and np.array_equal(s.cpu().numpy(), want[1])
