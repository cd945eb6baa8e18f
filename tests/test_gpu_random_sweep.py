"""Seeded random sweep over the entry points, bit for bit against the oracle.

Each case draws its own shape (empty, tiny, ragged, several tiles), format,
input type, scale (including extreme ones) and an offset that makes the input
start off a 16-byte boundary, so that every kernel's fast and guarded paths
and their edges meet values the hand-written cases do not.  The cases are
small; the sweep takes seconds.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq

from test_gpu_parity import dev_scalar, f32_bits, host_bits, with_specials

pytestmark = pytest.mark.gpu
E4M3, E5M2 = fq.E4M3, fq.E5M2
CASES = range(100)


def draw_tensor(rng, shape, dtype, dev):
    """Values over many binades, sometimes with Inf / NaN / zeros / subnormals,
    and sometimes as a view that starts 1-3 elements into its allocation."""
    n = int(np.prod(shape))
    off = int(rng.choice([0, 0, 0, 1, 3]))
    g = torch.Generator().manual_seed(int(rng.integers(1 << 30)))
    base = torch.randn(n + off, generator=g) * float(10.0 ** rng.uniform(-3, 4))
    if rng.random() < 0.4:
        base = base * torch.exp(3 * torch.randn(n + off, generator=g))
    t = base.to(dtype).to(dev)
    if n >= 16 and rng.random() < 0.25:
        t = with_specials(t, int(rng.integers(1 << 20)))
    return t[off:].view(shape)


def draw_scale(rng):
    r = rng.random()
    if r < 0.05:
        return np.float32(3.4028235e38)
    if r < 0.10:
        return np.float32(1.2e-38)
    return np.float32(10.0 ** rng.uniform(-6, 6))


def shape2(rng, hi=300):
    return int(rng.integers(1, hi)), int(rng.integers(1, hi))


@pytest.mark.parametrize("case", CASES)
def test_quantize_with_amax_and_count(cuda, oracle, case):
    rng = np.random.default_rng(1000 + case)
    n = int(rng.choice([0, 1, 7, 16, 17, int(rng.integers(1, 70000))]))
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    x = draw_tensor(rng, (n,), dtype, cuda)
    sc = draw_scale(rng)
    q = torch.empty(n, dtype=torch.uint8, device=cuda)
    am = torch.empty(1, device=cuda)
    sat = torch.empty(1, dtype=torch.int64, device=cuda)
    fq.fp8_quantize(x, fmt, dev_scalar(sc, cuda), q, am, sat)
    torch.cuda.synchronize()
    xb = host_bits(x)
    wq, wsat = oracle.quantize(xb, fmt, sc)
    assert np.array_equal(q.cpu().numpy(), wq)
    assert sat.item() == wsat
    assert f32_bits(am.item()) == f32_bits(oracle.amax(xb))


@pytest.mark.parametrize("case", CASES)
def test_cast_transpose(cuda, oracle, case):
    rng = np.random.default_rng(2000 + case)
    rows, cols = shape2(rng)
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    x = draw_tensor(rng, (rows, cols), dtype, cuda)
    sc = draw_scale(rng)
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    am = torch.empty(1, device=cuda)
    fq.fp8_quantize_cast_transpose(x, fmt, dev_scalar(sc, cuda), q_row, q_col, am)
    torch.cuda.synchronize()
    xb = host_bits(x)
    wr, wc = oracle.cast_transpose(xb, fmt, sc)
    assert np.array_equal(q_row.cpu().numpy(), wr) and np.array_equal(q_col.cpu().numpy(), wc)
    assert f32_bits(am.item()) == f32_bits(oracle.amax(xb))


@pytest.mark.parametrize("case", CASES)
def test_block_quantize(cuda, oracle, case):
    rng = np.random.default_rng(3000 + case)
    rows, cols = shape2(rng, 400)
    br = 128 if rng.random() < 0.5 else 1
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    x = draw_tensor(rng, (rows, cols), dtype, cuda)
    q = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    si = torch.empty((-(-rows // br), -(-cols // 128)), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block(x, br, 128, fmt, q, si)
    torch.cuda.synchronize()
    wq, wsi = oracle.quantize_block(host_bits(x), br, 128, fmt)
    assert np.array_equal(q.cpu().numpy(), wq)
    assert np.array_equal(si.cpu().numpy().view(np.uint32), wsi.view(np.uint32))


@pytest.mark.parametrize("case", CASES)
def test_dequantize(cuda, oracle, case):
    rng = np.random.default_rng(4000 + case)
    rows, cols = shape2(rng, 400)
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    block = [(0, 0), (128, 128), (1, 128)][int(rng.integers(3))]
    out_bf16 = rng.random() < 0.6
    g = torch.Generator().manual_seed(case)
    q = torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.uint8)
    br, bc = block
    sshape = (1,) if br == 0 else (-(-rows // br), -(-cols // bc))
    si = torch.from_numpy(np.array([draw_scale(rng) for _ in range(int(np.prod(sshape)))],
                                   dtype=np.float32).reshape(sshape))
    y = torch.empty((rows, cols), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=cuda)
    fq.fp8_dequantize(q.to(cuda), fmt, si.to(cuda), y, br, bc)
    torch.cuda.synchronize()
    want = oracle.dequantize(q.numpy(), fmt, si.numpy(), br, bc, out_dt=oracle.BF16 if out_bf16 else oracle.FP32)
    got = host_bits(y)
    if out_bf16:
        assert np.array_equal(got, want)
    else:
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("case", CASES)
def test_current_scaling_call(cuda, oracle, case):
    rng = np.random.default_rng(5000 + case)
    n = int(rng.choice([0, 5, 4096, int(rng.integers(1, 3_000_000))]))
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    margin = int(rng.integers(-3, 4))
    x = draw_tensor(rng, (n,), dtype, cuda)
    q = torch.empty(n, dtype=torch.uint8, device=cuda)
    am, s, si = (torch.empty(1, device=cuda) for _ in range(3))
    fq.fp8_quantize_current(x, fmt, q, margin, am, s, si)
    torch.cuda.synchronize()
    xb = host_bits(x)
    wa = oracle.amax(xb)
    ws, wsi = oracle.compute_scale(wa, fmt, margin)
    assert f32_bits(am.item()) == f32_bits(wa)
    assert (f32_bits(s.item()), f32_bits(si.item())) == (f32_bits(ws), f32_bits(wsi))
    assert np.array_equal(q.cpu().numpy(), oracle.quantize(xb, fmt, ws)[0])


@pytest.mark.parametrize("case", CASES)
def test_mx_both_directions(cuda, oracle, case):
    rng = np.random.default_rng(6000 + case)
    if rng.random() < 0.5:  # the tile kernel's shapes: 32-row multiples, 128-column multiples
        rows, cols = 32 * int(rng.integers(1, 12)), 128 * int(rng.integers(1, 4))
    else:
        rows, cols = shape2(rng)
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    x = draw_tensor(rng, (rows, cols), dtype, cuda)
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    s_row = torch.empty((rows, -(-cols // 32)), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    s_col = torch.empty((cols, -(-rows // 32)), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_mx(x, fmt, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    xb = host_bits(x)
    wq, ws = oracle.quantize_mx(xb, fmt)
    assert np.array_equal(s_row.cpu().numpy(), ws) and np.array_equal(q_row.cpu().numpy(), wq)
    wq, ws = oracle.quantize_mx(np.ascontiguousarray(xb.T), fmt)
    assert np.array_equal(s_col.cpu().numpy(), ws) and np.array_equal(q_col.cpu().numpy(), wq)


@pytest.mark.parametrize("case", CASES)
def test_hybrid(cuda, oracle, case):
    rng = np.random.default_rng(7000 + case)
    rows, cols = shape2(rng)
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    f_row = E4M3 if rng.random() < 0.5 else E5M2
    f_col = E4M3 if rng.random() < 0.5 else E5M2
    from_deq = rng.random() < 0.5
    source = fq.COLUMNWISE_FROM_ROWWISE_DEQUANTIZED if from_deq else fq.COLUMNWISE_FROM_ORIGINAL
    x = draw_tensor(rng, (rows, cols), dtype, cuda)
    s_row, s_col = draw_scale(rng), draw_scale(rng)
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_hybrid(x, f_row, dev_scalar(s_row, cuda), q_row, f_col, dev_scalar(s_col, cuda), q_col, source)
    torch.cuda.synchronize()
    wr, wc = oracle.quantize_hybrid(host_bits(x), f_row, s_row, f_col, s_col, 1 if from_deq else 0)
    assert np.array_equal(q_row.cpu().numpy(), wr) and np.array_equal(q_col.cpu().numpy(), wc)


@pytest.mark.parametrize("case", CASES)
def test_block_cast_transpose(cuda, oracle, case):
    rng = np.random.default_rng(8000 + case)
    if rng.random() < 0.5:  # the tile kernel's shapes
        rows, cols = 128 * int(rng.integers(1, 4)), 128 * int(rng.integers(1, 4))
    else:
        rows, cols = shape2(rng)
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    x = draw_tensor(rng, (rows, cols), dtype, cuda)
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    si_row = torch.empty((rows, -(-cols // 128)), dtype=torch.float32, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    si_col = torch.empty((cols, -(-rows // 128)), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block_cast_transpose(x, fmt, q_row, si_row, q_col, si_col)
    torch.cuda.synchronize()
    xb = host_bits(x)
    wq, wsi = oracle.quantize_block(xb, 1, 128, fmt)
    assert np.array_equal(q_row.cpu().numpy(), wq)
    assert np.array_equal(si_row.cpu().numpy().view(np.uint32), wsi.view(np.uint32))
    wq, wsi = oracle.quantize_block(np.ascontiguousarray(xb.T), 1, 128, fmt)
    assert np.array_equal(q_col.cpu().numpy(), wq)
    assert np.array_equal(si_col.cpu().numpy().view(np.uint32), wsi.view(np.uint32))


@pytest.mark.parametrize("case", range(20))
def test_delayed_sequence(cuda, oracle, case):
    rng = np.random.default_rng(9000 + case)
    L = int(rng.choice([1, 2, 3, 1000, 1024, int(rng.integers(1, 5000))]))
    algo = fq.AMAX_MAX if rng.random() < 0.6 else fq.AMAX_MOST_RECENT
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    margin = int(rng.integers(-2, 3))
    hist = torch.zeros(L, device=cuda)
    h_ref = np.zeros(L, dtype=np.float32)
    s, si = dev_scalar(np.float32(1.0), cuda), dev_scalar(np.float32(1.0), cuda)
    ws = np.float32(1.0)
    step0 = int(rng.integers(0, 1 << 40))
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    for k in range(step0, step0 + 5):
        n = int(rng.integers(0, 50000))
        x = draw_tensor(rng, (n,), dtype, cuda)
        q = torch.empty(n, dtype=torch.uint8, device=cuda)
        am = torch.empty(1, device=cuda)
        sat = torch.empty(1, dtype=torch.int64, device=cuda)
        fq.fp8_quantize_delayed(x, fmt, s, si, q, hist, k, algo, margin, am, sat)
        torch.cuda.synchronize()
        xb = host_bits(x)
        wq, wsat = oracle.quantize(xb, fmt, ws)
        assert np.array_equal(q.cpu().numpy(), wq) and sat.item() == wsat, k
        wa = oracle.amax(xb)
        assert f32_bits(am.item()) == f32_bits(wa), k
        ws, wsi = oracle.update_delayed(h_ref, k, wa, algo, fmt, margin)
        assert (f32_bits(s.item()), f32_bits(si.item())) == (f32_bits(ws), f32_bits(wsi)), k
        assert np.array_equal(hist.cpu().numpy().view(np.uint32), h_ref.view(np.uint32)), k


@pytest.mark.parametrize("case", range(30))
def test_grouped(cuda, oracle, case):
    rng = np.random.default_rng(10000 + case)
    count = int(rng.choice([1, 2, 5, 33, int(rng.integers(1, 129))]))
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    margin = int(rng.integers(-2, 3))
    xs = []
    for _ in range(count):
        n = int(rng.choice([0, 1, 8, 4096, int(rng.integers(1, 40000))]))
        x = draw_tensor(rng, (n + 8,), dtype, cuda)  # grouped tensors must be 16-byte aligned:
        xs.append(x.contiguous()[:n] if x.data_ptr() % 16 == 0 else x.clone()[:n])  # re-based copies
    am, s, si = (torch.empty(count, device=cuda) for _ in range(3))
    fq.fp8_amax_grouped(xs, am, fmt, margin, s, si)
    qs = [torch.empty(x.shape, dtype=torch.uint8, device=cuda) for x in xs]
    fq.fp8_quantize_grouped(xs, fmt, s, qs)
    torch.cuda.synchronize()
    for i, x in enumerate(xs):
        xb = host_bits(x)
        wa = oracle.amax(xb)
        ws, wsi = oracle.compute_scale(wa, fmt, margin)
        assert f32_bits(am[i].item()) == f32_bits(wa), i
        assert (f32_bits(s[i].item()), f32_bits(si[i].item())) == (f32_bits(ws), f32_bits(wsi)), i
        assert np.array_equal(qs[i].cpu().numpy(), oracle.quantize(xb, fmt, ws)[0]), i


@pytest.mark.parametrize("case", CASES)
def test_mx_dequantize(cuda, oracle, case):
    rng = np.random.default_rng(11000 + case)
    rows, cols = shape2(rng, 200)
    if rng.random() < 0.5:
        cols = 32 * int(rng.integers(1, 8))  # the vector kernel's shapes
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    out_bf16 = rng.random() < 0.6
    g = torch.Generator().manual_seed(11000 + case)
    q = torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.uint8)
    sc = torch.randint(0, 256, (rows, -(-cols // 32)), generator=g, dtype=torch.uint8)
    y = torch.empty((rows, cols), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=cuda)
    fq.fp8_dequantize_mx(q.to(cuda), sc.to(cuda), fmt, y)
    torch.cuda.synchronize()
    want = oracle.dequantize_mx(q.numpy(), sc.numpy(), fmt, out_dt=oracle.BF16 if out_bf16 else oracle.FP32)
    got = host_bits(y)
    if out_bf16:
        assert np.array_equal(got, want)
    else:
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("case", range(30))
def test_block128_scales_to_mx(cuda, oracle, case):
    rng = np.random.default_rng(12000 + case)
    rows, cols = shape2(rng, 700)
    nbr, nbc = -(-rows // 128), -(-cols // 128)
    k = rng.integers(-140, 130, size=(nbr, nbc))
    si = np.ldexp(np.float32(1.0), k).astype(np.float32)
    odd = rng.random((nbr, nbc)) < 0.1
    si[odd] = np.float32(3.0)  # not a power of two
    out = torch.empty((rows, -(-cols // 32)), dtype=torch.uint8, device=cuda)
    bad = torch.empty(1, dtype=torch.int64, device=cuda)
    fq.fp8_block128_scales_to_mx(torch.from_numpy(si).to(cuda), rows, cols, out, bad)
    torch.cuda.synchronize()
    want, wbad = oracle.block128_scales_to_mx(si, rows, cols)
    assert np.array_equal(out.cpu().numpy(), want) and bad.item() == wbad


@pytest.mark.parametrize("case", CASES)
def test_amax_and_scale(cuda, oracle, case):
    rng = np.random.default_rng(13000 + case)
    n = int(rng.choice([0, 1, 3, 9, 4096, int(rng.integers(1, 4_000_000))]))
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    margin = int(rng.integers(-5, 6))
    x = draw_tensor(rng, (n,), dtype, cuda)
    am, s, si = (torch.empty(1, device=cuda) for _ in range(3))
    if rng.random() < 0.5 and n <= (1 << 28):
        fq.fp8_amax_noalloc(x, am, fmt, margin, s, si)
    else:
        fq.fp8_amax(x, am, fmt, margin, s, si)
    torch.cuda.synchronize()
    wa = oracle.amax(host_bits(x))
    ws, wsi = oracle.compute_scale(wa, fmt, margin)
    assert f32_bits(am.item()) == f32_bits(wa)
    assert (f32_bits(s.item()), f32_bits(si.item())) == (f32_bits(ws), f32_bits(wsi))


@pytest.mark.parametrize("case", range(30))
def test_update_scale_delayed(cuda, oracle, case):
    rng = np.random.default_rng(14000 + case)
    L = int(rng.choice([1, 2, 31, 32, 33, 1024, 65536, int(rng.integers(1, 70000) % 65536 + 1)]))
    algo = fq.AMAX_MAX if rng.random() < 0.6 else fq.AMAX_MOST_RECENT
    fmt = E4M3 if rng.random() < 0.5 else E5M2
    margin = int(rng.integers(-3, 4))
    h0 = (rng.random(L) * float(10.0 ** rng.uniform(-3, 3))).astype(np.float32)
    if rng.random() < 0.2:
        h0[int(rng.integers(L))] = np.float32("nan")
    hist, h_ref = torch.from_numpy(h0.copy()).to(cuda), h0.copy()
    s, si = torch.empty(1, device=cuda), torch.empty(1, device=cuda)
    for _ in range(4):
        step = int(rng.integers(0, 1 << 45))
        new = None if rng.random() < 0.2 else np.float32(10.0 ** rng.uniform(-4, 4))
        fq.fp8_update_scale_delayed(hist, step, None if new is None else dev_scalar(new, cuda), algo, fmt, margin,
                                    s, si)
        torch.cuda.synchronize()
        ws, wsi = oracle.update_delayed(h_ref, step, new, algo, fmt, margin)
        assert (f32_bits(s.item()), f32_bits(si.item())) == (f32_bits(ws), f32_bits(wsi)), step
        assert np.array_equal(hist.cpu().numpy().view(np.uint32), h_ref.view(np.uint32)), step
