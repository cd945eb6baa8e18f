"""GPU parity: the sm_103a library (called through its C ABI) against the CPU
oracle, element by element, on the same seeded bytes.

Bar: FP8 codes, saturation counts, amax, scale, scale_inv and dequantized
values are compared bit for bit (both sides compute fl32(x * scale) and one
round-to-nearest-even conversion, so there is nothing to tolerate).
Sizes span several tiles with ragged tails; edge cases cover empty inputs,
unaligned pointers, Inf / NaN / signed zeros / subnormals, and the full-size
workloads of the benchmark.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq
from fp8_scaled_quantization_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

E4M3, E5M2 = fq.E4M3, fq.E5M2
FMTS = [E4M3, E5M2]


# ------------------------------------------------------------------ helpers

def host_bits(x: torch.Tensor) -> np.ndarray:
    """Bit pattern of a device tensor as numpy (uint16 for BF16, float32 for fp32)."""
    h = x.detach().contiguous().cpu()
    if h.dtype == torch.bfloat16:
        return h.view(torch.int16).numpy().view(np.uint16)
    return h.numpy()


def f32_bits(v) -> int:
    return int(np.float32(v).view(np.uint32))


def dev_scalar(v: float, dev) -> torch.Tensor:
    return torch.tensor([v], dtype=torch.float32, device=dev)


def random_input(n_or_shape, dtype, seed, dev, spread=True):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(n_or_shape, generator=g) * 40
    if spread:
        x = x * torch.exp(3 * torch.randn(n_or_shape, generator=g))
    return x.to(dtype).to(dev)


def with_specials(x: torch.Tensor, seed: int) -> torch.Tensor:
    """Plant Inf, -Inf, NaN, +-0, subnormals and huge values at random places."""
    flat = x.view(-1)
    n = flat.numel()
    if n < 16:
        return x
    g = torch.Generator(device="cpu").manual_seed(seed)
    pos = torch.randperm(n, generator=g)[:12].to(x.device)
    vals = torch.tensor([float("inf"), -float("inf"), float("nan"), 0.0, -0.0, 1e-40, -1e-39, 3e38, -3e38,
                         2.5e-45, 65504.0, -1e30], dtype=torch.float32)
    flat[pos] = vals.to(x.dtype).to(x.device)
    return x


def quantize_gpu(x, fmt, scale, want_amax=True, want_sat=True):
    dev = x.device
    q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    am = torch.empty(1, dtype=torch.float32, device=dev) if want_amax else None
    sat = torch.empty(1, dtype=torch.int64, device=dev) if want_sat else None
    s = dev_scalar(scale, dev)
    fq.fp8_quantize(x, fmt, s, q, am, sat)
    torch.cuda.synchronize()
    return q, am, sat


# ---------------------------------------------------------------- amax / scale

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n", [0, 1, 7, 15, 16, 17, 1000, 4097, (1 << 20) + 3])
def test_amax_and_current_scale(cuda, oracle, dtype, n):
    x = random_input(n, dtype, 100 + n, cuda)
    xb = host_bits(x)
    want_amax = oracle.amax(xb)
    for fmt in FMTS:
        for margin in (0, 1, 3):
            am, s, si = (torch.empty(1, dtype=torch.float32, device=cuda) for _ in range(3))
            fq.fp8_amax(x, am, fmt, margin, s, si)
            torch.cuda.synchronize()
            ws, wsi = oracle.compute_scale(want_amax, fmt, margin)
            assert f32_bits(am.item()) == f32_bits(want_amax)
            assert (f32_bits(s.item()), f32_bits(si.item())) == (f32_bits(ws), f32_bits(wsi))


@pytest.mark.parametrize("offset", [1, 3, 5])
def test_amax_unaligned_and_specials(cuda, oracle, offset):
    base = random_input(50_000, torch.bfloat16, 7, cuda)
    x = base[offset:]  # not 16-byte aligned
    am = torch.empty(1, dtype=torch.float32, device=cuda)
    fq.fp8_amax(x, am)
    torch.cuda.synchronize()
    assert f32_bits(am.item()) == f32_bits(oracle.amax(host_bits(x)))
    y = x.clone()
    y[123] = float("inf")
    fq.fp8_amax(y, am)
    torch.cuda.synchronize()
    assert am.item() == float("inf")
    y[4567] = float("nan")
    s, si = torch.empty(1, device=cuda), torch.empty(1, device=cuda)
    fq.fp8_amax(y, am, E4M3, 0, s, si)
    torch.cuda.synchronize()
    assert f32_bits(am.item()) == 0x7FC00000
    assert s.item() == 1.0 and si.item() == 1.0


def test_amax_zero_tensor_gives_scale_one(cuda):
    x = torch.zeros(12345, dtype=torch.bfloat16, device=cuda)
    am, s, si = (torch.full((1,), 7.0, device=cuda) for _ in range(3))
    fq.fp8_amax(x, am, E4M3, 0, s, si)
    torch.cuda.synchronize()
    assert (am.item(), s.item(), si.item()) == (0.0, 1.0, 1.0)


# ---------------------------------------------------------------- quantize

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n", [0, 1, 5, 16, 31, 33, 8191, 100_003, 3 * (1 << 18) + 11])
def test_quantize_matches_oracle(cuda, oracle, dtype, fmt, n):
    x = with_specials(random_input(n, dtype, 200 + n, cuda), n)
    xb = host_bits(x)
    scale = np.float32(0.37)
    q, am, sat = quantize_gpu(x, fmt, scale)
    wq, wsat = oracle.quantize(xb, fmt, scale)
    assert np.array_equal(q.cpu().numpy(), wq)
    assert sat.item() == wsat
    assert f32_bits(am.item()) == f32_bits(oracle.amax(xb))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("scale", [1.0, 2.0 ** -20, 3.0, 448.0 / 2000.0, 1e30])
def test_all_bf16_patterns(cuda, oracle, fmt, scale):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(cuda)
    for want_amax, want_sat in [(False, False), (True, True), (False, True)]:
        q, am, sat = quantize_gpu(x, fmt, scale, want_amax, want_sat)
        wq, wsat = oracle.quantize(bits, fmt, np.float32(scale))
        assert np.array_equal(q.cpu().numpy(), wq)
        if want_sat:
            assert sat.item() == wsat
        if want_amax:
            assert f32_bits(am.item()) == 0x7FC00000  # the patterns include NaN


@pytest.mark.parametrize("fmt", FMTS)
def test_nan_and_inf_codes(cuda, fmt):
    x = torch.tensor([float("nan"), -float("nan"), float("inf"), -float("inf"), -0.0, 0.0] * 8,
                     dtype=torch.bfloat16, device=cuda)
    q, _, _ = quantize_gpu(x, fmt, 1.0, False, False)
    q = q.cpu().tolist()[:6]
    inf = 0x7C if fmt == E5M2 else 0x7E
    assert q == [0x7F, 0x7F, inf, 0x80 | inf, 0x80, 0x00]


@pytest.mark.parametrize("offset", [1, 2, 9])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_unaligned(cuda, oracle, offset, dtype):
    base = with_specials(random_input(70_001, dtype, 31, cuda), 5)
    x = base[offset:]
    qbase = torch.empty(70_001 + 16, dtype=torch.uint8, device=cuda)
    q = qbase[3:3 + x.numel()]  # unaligned output too
    am = torch.empty(1, device=cuda)
    sat = torch.empty(1, dtype=torch.int64, device=cuda)
    fq.fp8_quantize(x, E4M3, dev_scalar(0.5, cuda), q, am, sat)
    torch.cuda.synchronize()
    wq, wsat = oracle.quantize(host_bits(x), E4M3, np.float32(0.5))
    assert np.array_equal(q.cpu().numpy(), wq)
    assert sat.item() == wsat


def test_quantize_does_not_write_outside(cuda, oracle):
    x = random_input(1000, torch.bfloat16, 3, cuda)
    buf = torch.full((1000 + 64,), 0xAB, dtype=torch.uint8, device=cuda)
    q = buf[32:32 + 1000]
    fq.fp8_quantize(x, E4M3, dev_scalar(1.0, cuda), q)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:32] == 0xAB) and np.all(b[-32:] == 0xAB)


# ---------------------------------------------------------- cast-transpose

CT_SHAPES = [(128, 128), (256, 384), (384, 128), (130, 200), (16, 16), (1, 1), (0, 5), (5, 0), (333, 17),
             (48, 1040), (1040, 48)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", CT_SHAPES)
def test_cast_transpose_matches_oracle(cuda, oracle, dtype, fmt, shape):
    x = with_specials(random_input(shape, dtype, sum(shape), cuda), 1)
    rows, cols = shape
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    am = torch.empty(1, device=cuda)
    s = np.float32(1.75)
    fq.fp8_quantize_cast_transpose(x, fmt, dev_scalar(s, cuda), q_row, q_col, am)
    torch.cuda.synchronize()
    xb = host_bits(x)
    wr, wc = oracle.cast_transpose(xb, fmt, s)
    assert np.array_equal(q_row.cpu().numpy(), wr)
    assert np.array_equal(q_col.cpu().numpy(), wc)
    assert f32_bits(am.item()) == f32_bits(oracle.amax(xb))


@pytest.mark.parametrize("which", ["row", "col"])
def test_cast_transpose_single_direction(cuda, oracle, which):
    x = random_input((256, 512), torch.bfloat16, 9, cuda)
    q = torch.empty((256, 512) if which == "row" else (512, 256), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_cast_transpose(x, E5M2, dev_scalar(0.01, cuda), q if which == "row" else None,
                                   q if which == "col" else None)
    torch.cuda.synchronize()
    wr, wc = oracle.cast_transpose(host_bits(x), E5M2, np.float32(0.01))
    assert np.array_equal(q.cpu().numpy(), wr if which == "row" else wc)


# --------------------------------------------------------------- blockwise

BLOCK_SHAPES = [(128, 128), (256, 384), (300, 260), (1, 1), (129, 1), (7, 1000), (64, 256)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("block", [(128, 128), (1, 128)])
@pytest.mark.parametrize("shape", BLOCK_SHAPES)
def test_block_quantize_matches_oracle(cuda, oracle, dtype, fmt, block, shape):
    g = torch.Generator(device="cpu").manual_seed(sum(shape) + block[0])
    br, bc = block
    nbr, nbc = -(-shape[0] // br), -(-shape[1] // bc)
    mags = torch.exp(2 * torch.randn((nbr, nbc), generator=g))
    mags = mags.repeat_interleave(br, 0)[:shape[0]].repeat_interleave(bc, 1)[:, :shape[1]]
    x = (torch.randn(shape, generator=g) * mags).to(dtype).to(cuda)
    if x.numel() > 1000:
        x = with_specials(x, 2)
    q = torch.empty(shape, dtype=torch.uint8, device=cuda)
    si = torch.empty((nbr, nbc), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block(x, br, bc, fmt, q, si)
    torch.cuda.synchronize()
    wq, wsi = oracle.quantize_block(host_bits(x), br, bc, fmt)
    assert np.array_equal(si.cpu().numpy().view(np.uint32), wsi.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), wq)


# --------------------------------------------------------------- dequantize

@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(1, 1), (3, 7), (64, 256), (257, 129), (128, 4096)])
@pytest.mark.parametrize("block", [(0, 0), (128, 128), (1, 128)])
def test_dequantize_matches_oracle(cuda, oracle, out_dtype, fmt, shape, block):
    g = torch.Generator(device="cpu").manual_seed(shape[0] * 7 + shape[1])
    q = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
    br, bc = block
    nsi = (1, 1) if br == 0 else (-(-shape[0] // br), -(-shape[1] // bc))
    si = (torch.rand(nsi, generator=g) * 10 + 1e-3).to(torch.float32)
    y = torch.empty(shape, dtype=out_dtype, device=cuda)
    fq.fp8_dequantize(q.to(cuda), fmt, si.to(cuda), y, br, bc)
    torch.cuda.synchronize()
    want = oracle.dequantize(q.numpy(), fmt, si.numpy(), br, bc,
                             out_dt=oracle.BF16 if out_dtype == torch.bfloat16 else oracle.FP32)
    got = host_bits(y) if out_dtype == torch.bfloat16 else host_bits(y).view(np.uint32)
    want = want if out_dtype == torch.bfloat16 else want.view(np.uint32)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("offset", [1, 6])
def test_dequantize_unaligned_1d(cuda, oracle, offset):
    g = torch.Generator(device="cpu").manual_seed(offset)
    qb = torch.randint(0, 256, (10_000,), generator=g, dtype=torch.uint8).to(cuda)
    q = qb[offset:]
    y = torch.empty(q.numel(), dtype=torch.bfloat16, device=cuda)
    si = dev_scalar(0.125, cuda)
    fq.fp8_dequantize(q, E4M3, si, y)
    torch.cuda.synchronize()
    want = oracle.dequantize(q.cpu().numpy(), E4M3, np.array([0.125], np.float32)).ravel()
    assert np.array_equal(host_bits(y), want)


# --------------------------------------------------------- delayed scaling

@pytest.mark.parametrize("algo", [fq.AMAX_MAX, fq.AMAX_MOST_RECENT])
@pytest.mark.parametrize("hist_len", [1, 4, 1024])
def test_delayed_sequence_matches_oracle(cuda, oracle, algo, hist_len):
    steps, shape = 12, (96, 160)
    hist = torch.zeros(hist_len, dtype=torch.float32, device=cuda)
    s, si = torch.empty(1, device=cuda), torch.empty(1, device=cuda)
    am = torch.empty(1, device=cuda)
    sat = torch.empty(1, dtype=torch.int64, device=cuda)
    h_ref = np.zeros(hist_len, dtype=np.float32)
    fq.fp8_update_scale_delayed(hist, 0, None, algo, E4M3, 0, s, si)
    ws, wsi = oracle.update_delayed(h_ref, 0, None, algo, E4M3, 0)
    for k, x in enumerate(wl.w3_steps(shape=shape, steps=steps, device=cuda)):
        q = torch.empty(shape, dtype=torch.uint8, device=cuda)
        fq.fp8_quantize(x, E4M3, s, q, am, sat)
        fq.fp8_update_scale_delayed(hist, k, am, algo, E4M3, 0, s, si)
        torch.cuda.synchronize()
        xb = host_bits(x)
        wq, wsat = oracle.quantize(xb, E4M3, ws)
        assert np.array_equal(q.cpu().numpy(), wq), k
        assert sat.item() == wsat
        a = oracle.amax(xb)
        assert f32_bits(am.item()) == f32_bits(a)
        ws, wsi = oracle.update_delayed(h_ref, k, a, algo, E4M3, 0)
        assert (f32_bits(s.item()), f32_bits(si.item())) == (f32_bits(ws), f32_bits(wsi))
        assert np.array_equal(hist.cpu().numpy().view(np.uint32), h_ref.view(np.uint32))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("algo", [fq.AMAX_MAX, fq.AMAX_MOST_RECENT])
@pytest.mark.parametrize("hist_len,shape", [(1, (96, 160)), (4, (33, 77)), (1024, (96, 160))])
def test_fused_delayed_sequence_matches_oracle(cuda, oracle, dtype, algo, hist_len, shape):
    steps, margin, fmt = 10, 1, E5M2
    hist = torch.zeros(hist_len, dtype=torch.float32, device=cuda)
    s, si = torch.empty(1, device=cuda), torch.empty(1, device=cuda)
    am = torch.empty(1, device=cuda)
    sat = torch.empty(1, dtype=torch.int64, device=cuda)
    h_ref = np.zeros(hist_len, dtype=np.float32)
    fq.fp8_update_scale_delayed(hist, 0, None, algo, fmt, margin, s, si)
    ws, wsi = oracle.update_delayed(h_ref, 0, None, algo, fmt, margin)
    g = torch.Generator(device="cpu").manual_seed(hist_len)
    for k in range(steps):
        x = (torch.randn(shape, generator=g) * 1e-3 * 1.5 ** k).to(dtype).to(cuda)
        if k == 6:
            x.view(-1)[5] = float("inf")
        q = torch.empty(shape, dtype=torch.uint8, device=cuda)
        fq.fp8_quantize_delayed(x, fmt, s, si, q, hist, k, algo, margin, am, sat)
        torch.cuda.synchronize()
        xb = host_bits(x)
        wq, wsat = oracle.quantize(xb, fmt, ws)
        assert np.array_equal(q.cpu().numpy(), wq), k
        assert sat.item() == wsat
        a = oracle.amax(xb)
        assert f32_bits(am.item()) == f32_bits(a)
        ws, wsi = oracle.update_delayed(h_ref, k, a, algo, fmt, margin)
        assert (f32_bits(s.item()), f32_bits(si.item())) == (f32_bits(ws), f32_bits(wsi)), k
        assert np.array_equal(hist.cpu().numpy().view(np.uint32), h_ref.view(np.uint32))


def test_fused_delayed_unaligned(cuda, oracle):
    base = random_input(10_001, torch.bfloat16, 5, cuda)
    x = base[1:]
    hist = torch.zeros(8, device=cuda)
    s, si = dev_scalar(0.25, cuda), torch.empty(1, device=cuda)
    q = torch.empty(x.numel(), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_delayed(x, E4M3, s, si, q, hist, 3, fq.AMAX_MAX, 0)
    torch.cuda.synchronize()
    xb = host_bits(x)
    assert np.array_equal(q.cpu().numpy(), oracle.quantize(xb, E4M3, np.float32(0.25))[0])
    h = np.zeros(8, np.float32)
    ws, wsi = oracle.update_delayed(h, 3, oracle.amax(xb), oracle.ALGO_MAX, E4M3, 0)
    assert (s.item(), si.item()) == (float(ws), float(wsi))


def test_current_equals_delayed_history_one(cuda):
    x = random_input(33_333, torch.bfloat16, 4, cuda)
    am, s1, si1, s2, si2 = (torch.empty(1, device=cuda) for _ in range(5))
    hist = torch.zeros(1, device=cuda)
    for margin in (0, 2):
        fq.fp8_amax(x, am, E5M2, margin, s1, si1)
        fq.fp8_update_scale_delayed(hist, 5, am, fq.AMAX_MOST_RECENT, E5M2, margin, s2, si2)
        torch.cuda.synchronize()
        assert (s1.item(), si1.item()) == (s2.item(), si2.item())


def test_delayed_nan_history(cuda):
    hist = torch.tensor([1.0, float("nan"), 3.0], device=cuda)
    s, si = torch.empty(1, device=cuda), torch.empty(1, device=cuda)
    fq.fp8_update_scale_delayed(hist, 0, None, fq.AMAX_MAX, E4M3, 0, s, si)
    torch.cuda.synchronize()
    assert (s.item(), si.item()) == (1.0, 1.0)


# ----------------------------------------------- streams, graphs, workspace

@pytest.mark.parametrize("fused", [False, True])
def test_delayed_history_at_its_limit(cuda, oracle, fused):
    """A 65536-entry history (the largest accepted) prefilled with amaxes, and
    step numbers past 2^40, so the slot is a 64-bit remainder and the window
    maximum runs over every entry but the slot."""
    L = 65536
    g = torch.Generator(device="cpu").manual_seed(41)
    h0 = (torch.rand(L, generator=g) * 300).float()
    h0[12345] = 2500.0  # the window maximum, until its slot is overwritten
    hist, h_ref = h0.to(cuda), h0.numpy().copy()
    s, si = dev_scalar(np.float32(1.0), cuda), dev_scalar(np.float32(1.0), cuda)
    ws = np.float32(1.0)
    base = (1 << 40) + 12345 - 2 - ((1 << 40) % L)  # slots 12343, 12344, 12345, 12346
    for i, k in enumerate(range(base, base + 4)):
        x = random_input((64, 96), torch.bfloat16, 300 + i, cuda, spread=False)  # amax ~160 < the history's
        xb = host_bits(x)
        a = oracle.amax(xb)
        if fused:
            q = torch.empty(x.shape, dtype=torch.uint8, device=cuda)
            fq.fp8_quantize_delayed(x, E4M3, s, si, q, hist, k, fq.AMAX_MAX, 0)
        else:
            am = dev_scalar(a, cuda)
            fq.fp8_update_scale_delayed(hist, k, am, fq.AMAX_MAX, E4M3, 0, s, si)
        torch.cuda.synchronize()
        if fused:
            wq, _ = oracle.quantize(xb, E4M3, ws)
            assert np.array_equal(q.cpu().numpy(), wq), k
        ws, wsi = oracle.update_delayed(h_ref, k, a, fq.AMAX_MAX, E4M3, 0)
        assert (f32_bits(s.item()), f32_bits(si.item())) == (f32_bits(ws), f32_bits(wsi)), k
        assert np.array_equal(hist.cpu().numpy().view(np.uint32), h_ref.view(np.uint32)), k


def test_delayed_resume_from_a_saved_state(cuda):
    """Checkpoint / resume: all delayed-scaling state lives in caller buffers,
    so 8 steps, a host copy of history / scale / scale_inv, a restore into
    fresh device buffers and steps 8-15 give the codes, scales and history of
    an uninterrupted 16-step run, bit for bit."""
    xs = list(wl.w3_steps(shape=(96, 160), steps=16, device=cuda))

    def fresh():
        return torch.zeros(16, device=cuda), dev_scalar(np.float32(1.0), cuda), dev_scalar(np.float32(1.0), cuda)

    def run(state, steps):
        hist, s, si = state
        qs = []
        for k in steps:
            q = torch.empty(xs[k].shape, dtype=torch.uint8, device=cuda)
            fq.fp8_quantize_delayed(xs[k], E4M3, s, si, q, hist, k, fq.AMAX_MAX, 0)
            qs.append(q)
        return qs

    whole = fresh()
    q_whole = run(whole, range(16))
    first = fresh()
    q_first = run(first, range(8))
    saved = [t.cpu() for t in first]  # the checkpoint
    del first
    resumed = tuple(t.to(cuda) for t in saved)  # restored into new buffers
    q_rest = run(resumed, range(8, 16))
    torch.cuda.synchronize()
    for k, (a, b) in enumerate(zip(q_whole, q_first + q_rest)):
        assert torch.equal(a, b), k
    for a, b in zip(whole, resumed):
        assert np.array_equal(a.cpu().numpy().view(np.uint32), b.cpu().numpy().view(np.uint32))


def test_concurrent_host_threads_on_their_own_streams(cuda, oracle):
    """Four host threads, each with its own stream (and so its own workspace),
    call the library at the same time; ctypes drops the interpreter lock
    during the calls, so the workspace table and the error text are used
    concurrently."""
    import threading
    xs = [random_input(2_000_000, torch.bfloat16, 50 + i, cuda) * (i + 1) for i in range(4)]
    want = [oracle.amax(host_bits(x)) for x in xs]
    scales = [oracle.compute_scale(w, E4M3, 0)[0] for w in want]
    codes = [oracle.quantize(host_bits(x), E4M3, sc)[0] for x, sc in zip(xs, scales)]
    torch.cuda.synchronize()
    errors = []

    def work(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(10):
                    am, s, si = (torch.empty(1, device=cuda) for _ in range(3))
                    q = torch.empty(xs[i].shape, dtype=torch.uint8, device=cuda)
                    fq.fp8_amax(xs[i], am, E4M3, 0, s, si)
                    fq.fp8_quantize(xs[i], E4M3, s, q)
                    st.synchronize()
                    assert f32_bits(am.item()) == f32_bits(want[i]) and np.array_equal(q.cpu().numpy(), codes[i])
                    try:  # a 2 x 64 block is rejected in the library: this thread's error text
                        fq.fp8_quantize_block(xs[i][:256].view(2, 128), 2, 64, E4M3, q[:256].view(2, 128),
                                              torch.empty((1, 2), device=cuda))
                        raise AssertionError("a 2 x 64 block was accepted")
                    except fq.Fp8Error as e:
                        assert e.status == 2 and "block" in str(e), str(e)
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_two_streams_use_separate_workspaces(cuda, oracle):
    xa = random_input(3_000_000, torch.bfloat16, 11, cuda)
    xb = random_input(3_000_000, torch.bfloat16, 12, cuda) * 3
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for _ in range(20):
        ama, amb = torch.empty(1, device=cuda), torch.empty(1, device=cuda)
        with torch.cuda.stream(sa):
            fq.fp8_amax(xa, ama)
        with torch.cuda.stream(sb):
            fq.fp8_amax(xb, amb)
        outs.append((ama, amb))
    torch.cuda.synchronize()
    wa, wb = oracle.amax(host_bits(xa)), oracle.amax(host_bits(xb))
    for ama, amb in outs:
        assert (ama.item(), amb.item()) == (float(wa), float(wb))


def test_release_stream_workspace_and_reuse(cuda, oracle):
    """A stream's workspace is freed after its queued work and allocated again
    by the next reducing call; releasing twice, or a stream that never had
    one, is a no-op."""
    x = random_input(3_000_000, torch.bfloat16, 13, cuda)
    want = float(oracle.amax(host_bits(x)))
    st = torch.cuda.Stream()
    fq.release_stream_workspace(torch.cuda.Stream())
    for _ in range(3):
        am = torch.empty(1, device=cuda)
        with torch.cuda.stream(st):
            fq.fp8_amax(x, am)
            fq.release_stream_workspace(st)
            fq.release_stream_workspace(st)
        st.synchronize()
        assert am.item() == want


def test_cuda_graph_capture_and_replay(cuda, oracle):
    x = random_input((512, 768), torch.bfloat16, 21, cuda)
    am, s, si = (torch.empty(1, device=cuda) for _ in range(3))
    q_row = torch.empty((512, 768), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((768, 512), dtype=torch.uint8, device=cuda)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):  # first use of the capture stream happens inside the capture
        fq.fp8_amax(x, am, E4M3, 1, s, si)
        fq.fp8_quantize_cast_transpose(x, E4M3, s, q_row, q_col)
    for _ in range(3):
        x.mul_(1.5)
        graph.replay()
        torch.cuda.synchronize()
        xb = host_bits(x)
        ws, _ = oracle.compute_scale(oracle.amax(xb), E4M3, 1)
        assert s.item() == float(ws)
        wr, wc = oracle.cast_transpose(xb, E4M3, ws)
        assert np.array_equal(q_row.cpu().numpy(), wr) and np.array_equal(q_col.cpu().numpy(), wc)


def test_block_cast_transpose_in_a_captured_graph(cuda, oracle):
    """The tensor-map kernel captured once (its map, built on the host from
    x's address, is a kernel argument of the graph node) and replayed while x
    changes in place."""
    x = random_input((512, 768), torch.bfloat16, 23, cuda)
    q_row = torch.empty((512, 768), dtype=torch.uint8, device=cuda)
    s_row = torch.empty((512, 6), dtype=torch.float32, device=cuda)
    q_col = torch.empty((768, 512), dtype=torch.uint8, device=cuda)
    s_col = torch.empty((768, 4), dtype=torch.float32, device=cuda)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fq.fp8_quantize_block_cast_transpose(x, E4M3, q_row, s_row, q_col, s_col)
    for _ in range(3):
        x.mul_(1.5)
        graph.replay()
        torch.cuda.synchronize()
        xb = host_bits(x)
        wq, ws = oracle.quantize_block(xb, 1, 128, E4M3)
        assert np.array_equal(q_row.cpu().numpy(), wq) and np.array_equal(s_row.cpu().numpy(), ws)
        wqt, wst = oracle.quantize_block(np.ascontiguousarray(xb.T), 1, 128, E4M3)
        assert np.array_equal(q_col.cpu().numpy(), wqt) and np.array_equal(s_col.cpu().numpy(), wst)


def test_reducing_casts_in_a_captured_graph(cuda, oracle):
    """The reducing casts and their finalize replayed from a graph, with the
    stream workspace created inside the capture."""
    x = random_input(1_000_000, torch.bfloat16, 71, cuda)
    one = dev_scalar(np.float32(1.0), cuda)
    q = torch.empty(x.shape, dtype=torch.uint8, device=cuda)
    qd = torch.empty(x.shape, dtype=torch.uint8, device=cuda)
    am = torch.empty(1, device=cuda)
    sat = torch.empty(1, dtype=torch.int64, device=cuda)
    hist = torch.zeros(16, device=cuda)
    s, si = dev_scalar(np.float32(1.0), cuda), dev_scalar(np.float32(1.0), cuda)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fq.fp8_quantize(x, E4M3, one, q, am, sat)
        fq.fp8_quantize_delayed(x, E4M3, s, si, qd, hist, 3, fq.AMAX_MAX, 0)
    prev = np.float32(1.0)
    for _ in range(3):
        x.mul_(1.5)
        graph.replay()
        torch.cuda.synchronize()
        xb = host_bits(x)
        wq, wsat = oracle.quantize(xb, E4M3, np.float32(1.0))
        wam = oracle.amax(xb)
        assert np.array_equal(q.cpu().numpy(), wq) and sat.item() == wsat
        assert f32_bits(am.item()) == f32_bits(wam)
        wqd, _ = oracle.quantize(xb, E4M3, prev)
        assert np.array_equal(qd.cpu().numpy(), wqd)
        ws, wsi = oracle.compute_scale(wam, E4M3, 0)  # the other slots hold 0
        assert f32_bits(s.item()) == f32_bits(ws) and f32_bits(si.item()) == f32_bits(wsi)
        assert f32_bits(hist[3].item()) == f32_bits(wam)
        prev = ws


def test_launch_counter_counts_kernels(cuda):
    x = random_input(1000, torch.bfloat16, 1, cuda)
    q = torch.empty(1000, dtype=torch.uint8, device=cuda)
    before = fq.launch_count()
    fq.fp8_quantize(x, E4M3, dev_scalar(1.0, cuda), q)
    fq.fp8_dequantize(q, E4M3, dev_scalar(1.0, cuda), torch.empty(1000, dtype=torch.bfloat16, device=cuda))
    assert fq.launch_count() - before == 2


def test_errors_are_raised(cuda):
    x = random_input(100, torch.bfloat16, 1, cuda)
    q = torch.empty(100, dtype=torch.uint8, device=cuda)
    with pytest.raises(fq.Fp8Error):
        fq.fp8_quantize(x, 7, dev_scalar(1.0, cuda), q)
    with pytest.raises(fq.Fp8Error):
        fq.fp8_quantize_block(x.view(10, 10), 64, 64, E4M3, q.view(10, 10), torch.empty((1, 1), device=cuda))
    with pytest.raises(fq.Fp8Error):
        fq.fp8_update_scale_delayed(torch.zeros(0, device=cuda), 0, None, fq.AMAX_MAX, E4M3, 0,
                                    torch.empty(1, device=cuda), torch.empty(1, device=cuda))


# ---------------------------------------------------------------------------
# Blockwise cast + transpose (1 x 128 rowwise, 128 x 1 columnwise)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(256, 384), (128, 128), (130, 200), (1, 300), (384, 1)])
def test_block_cast_transpose_matches_oracle(cuda, oracle, dtype, fmt, shape):
    rows, cols = shape
    g = torch.Generator(device="cpu").manual_seed(rows * 7 + cols)
    x = (torch.randn(shape, generator=g) * torch.exp(2 * torch.randn((rows, 1), generator=g))
         * torch.exp(2 * torch.randn((1, cols), generator=g))).to(dtype).to(cuda)
    if x.numel() > 500:
        x = with_specials(x, 3)
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    s_row = torch.empty((rows, -(-cols // 128)), dtype=torch.float32, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    s_col = torch.empty((cols, -(-rows // 128)), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block_cast_transpose(x, fmt, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    xb = host_bits(x)
    wq, ws = oracle.quantize_block(xb, 1, 128, fmt)
    assert np.array_equal(s_row.cpu().numpy().view(np.uint32), ws.view(np.uint32))
    assert np.array_equal(q_row.cpu().numpy(), wq)
    wqt, wst = oracle.quantize_block(np.ascontiguousarray(xb.T), 1, 128, fmt)
    assert np.array_equal(s_col.cpu().numpy().view(np.uint32), wst.view(np.uint32))
    assert np.array_equal(q_col.cpu().numpy(), wqt)


@pytest.mark.parametrize("shape", [(128, 128), (384, 128), (1024, 12800), (2048, 20480)])
@pytest.mark.parametrize("direction", ["both", "rows", "cols"])
def test_block_cast_transpose_tile_ring(cuda, oracle, shape, direction):
    """The persistent kernel at tile counts that leave a consumer group idle
    (1 and 3 tiles), wrap the stage ring (800 tiles: 5 or 6 per CTA) and run
    16-17 tiles per CTA, with Inf / NaN planted in some tiles; no bounded wait
    inside the kernel gives up."""
    rows, cols = shape
    x = with_specials(random_input(shape, torch.bfloat16, rows + cols, cuda), rows)
    before = fq.wait_timeouts()
    want_rows, want_cols = direction != "cols", direction != "rows"
    q_row = torch.full((rows, cols), 0xAA, dtype=torch.uint8, device=cuda) if want_rows else None
    s_row = torch.zeros((rows, cols // 128), dtype=torch.float32, device=cuda) if want_rows else None
    q_col = torch.full((cols, rows), 0xAA, dtype=torch.uint8, device=cuda) if want_cols else None
    s_col = torch.zeros((cols, rows // 128), dtype=torch.float32, device=cuda) if want_cols else None
    fq.fp8_quantize_block_cast_transpose(x, E4M3, q_row, s_row, q_col, s_col)
    assert fq.wait_timeouts() == before
    xb = host_bits(x)
    if want_rows:
        wq, ws = oracle.quantize_block(xb, 1, 128, E4M3)
        assert np.array_equal(s_row.cpu().numpy().view(np.uint32), ws.view(np.uint32))
        assert np.array_equal(q_row.cpu().numpy(), wq)
    if want_cols:
        wqt, wst = oracle.quantize_block(np.ascontiguousarray(xb.T), 1, 128, E4M3)
        assert np.array_equal(s_col.cpu().numpy().view(np.uint32), wst.view(np.uint32))
        assert np.array_equal(q_col.cpu().numpy(), wqt)


@pytest.mark.parametrize("shape", [(256, 256), (1024, 12160)])
def test_block_cast_transpose_expired_waits_end_and_are_counted(cuda, oracle, native_lib, shape):
    """The bounded waits of the tiled path, made to expire: with the copy of
    each CTA's first tile skipped (test hook), the launch still ends (its
    consumers give up after their limit; with 760 tiles the copying thread
    also gives up on a stage that is never released), the expired waits are
    counted, and the next launch on the same context is exact again."""
    rows, cols = shape
    x = random_input(shape, torch.bfloat16, 31, cuda)
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    s_row = torch.empty((rows, cols // 128), dtype=torch.float32, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    s_col = torch.empty((cols, rows // 128), dtype=torch.float32, device=cuda)
    before = fq.wait_timeouts()
    assert native_lib.fp8_test_drop_tile_copy(0) == 0
    try:
        fq.fp8_quantize_block_cast_transpose(x, E4M3, q_row, s_row, q_col, s_col)
        expired = fq.wait_timeouts()
    finally:
        assert native_lib.fp8_test_drop_tile_copy(-1) == 0
    assert expired > before
    fq.fp8_quantize_block_cast_transpose(x, E4M3, q_row, s_row, q_col, s_col)
    assert fq.wait_timeouts() == expired
    xb = host_bits(x)
    wq, ws = oracle.quantize_block(xb, 1, 128, E4M3)
    assert np.array_equal(q_row.cpu().numpy(), wq) and np.array_equal(s_row.cpu().numpy(), ws)
    wqt, wst = oracle.quantize_block(np.ascontiguousarray(xb.T), 1, 128, E4M3)
    assert np.array_equal(q_col.cpu().numpy(), wqt) and np.array_equal(s_col.cpu().numpy(), wst)


def test_block_cast_transpose_tile_without_specials(cuda, oracle):
    """A 512 x 512 BF16 tensor with no Inf / NaN: every tile takes the paired
    two-value conversion of the columnwise codes."""
    g = torch.Generator(device="cpu").manual_seed(77)
    x = (torch.randn((512, 512), generator=g) * torch.exp(3 * torch.randn((1, 512), generator=g))).to(torch.bfloat16)
    x = x.to(cuda)
    q = torch.empty((512, 512), dtype=torch.uint8, device=cuda)
    s = torch.empty((512, 4), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block_cast_transpose(x, E5M2, None, None, q, s)
    torch.cuda.synchronize()
    wq, ws = oracle.quantize_block(np.ascontiguousarray(host_bits(x).T), 1, 128, E5M2)
    assert np.array_equal(q.cpu().numpy(), wq) and np.array_equal(s.cpu().numpy(), ws)


def test_block_cast_transpose_one_direction(cuda, oracle):
    x = random_input((256, 512), torch.bfloat16, 17, cuda)
    q = torch.empty((512, 256), dtype=torch.uint8, device=cuda)
    s = torch.empty((512, 2), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block_cast_transpose(x, E4M3, None, None, q, s)
    torch.cuda.synchronize()
    wq, ws = oracle.quantize_block(np.ascontiguousarray(host_bits(x).T), 1, 128, E4M3)
    assert np.array_equal(q.cpu().numpy(), wq) and np.array_equal(s.cpu().numpy(), ws)
    q2 = torch.empty((256, 512), dtype=torch.uint8, device=cuda)
    s2 = torch.empty((256, 4), dtype=torch.float32, device=cuda)
    fq.fp8_quantize_block_cast_transpose(x, E4M3, q2, s2)
    torch.cuda.synchronize()
    wq2, ws2 = oracle.quantize_block(host_bits(x), 1, 128, E4M3)
    assert np.array_equal(q2.cpu().numpy(), wq2) and np.array_equal(s2.cpu().numpy(), ws2)


# ---------------------------------------------------------------------------
# Hybrid per-direction quantization ("[Pytorch][Common] Hybrid quantization #2817")
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmts", [(E4M3, E5M2), (E5M2, E4M3), (E4M3, E4M3), (E5M2, E5M2)])
@pytest.mark.parametrize("source", [fq.COLUMNWISE_FROM_ORIGINAL, fq.COLUMNWISE_FROM_ROWWISE_DEQUANTIZED])
@pytest.mark.parametrize("shape", [(256, 384), (130, 200), (48, 16), (1, 1)])
def test_hybrid_matches_oracle(cuda, oracle, dtype, fmts, source, shape):
    fmt_row, fmt_col = fmts
    rows, cols = shape
    x = random_input(shape, dtype, rows * 31 + cols + source, cuda)
    if x.numel() > 500:
        x = with_specials(x, 5)
    # Scales that put part of the tensor past each format's maximum, so that both
    # the fast path and the saturating slow path run.
    s_row, s_col = np.float32(3.0e2), np.float32(0.37)
    q_row = torch.empty((rows, cols), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((cols, rows), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_hybrid(x, fmt_row, dev_scalar(s_row, cuda), q_row, fmt_col, dev_scalar(s_col, cuda), q_col,
                           source)
    torch.cuda.synchronize()
    wr, wc = oracle.quantize_hybrid(host_bits(x), fmt_row, s_row, fmt_col, s_col, source)
    assert np.array_equal(q_row.cpu().numpy(), wr)
    assert np.array_equal(q_col.cpu().numpy(), wc)


def test_hybrid_same_format_and_scale_is_cast_transpose(cuda):
    x = random_input((384, 512), torch.bfloat16, 41, cuda)
    s = dev_scalar(np.float32(17.0), cuda)
    q_row = torch.empty((384, 512), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((512, 384), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_hybrid(x, E4M3, s, q_row, E4M3, s, q_col, fq.COLUMNWISE_FROM_ORIGINAL)
    r2 = torch.empty_like(q_row)
    c2 = torch.empty_like(q_col)
    fq.fp8_quantize_cast_transpose(x, E4M3, s, r2, c2)
    torch.cuda.synchronize()
    assert torch.equal(q_row, r2) and torch.equal(q_col, c2)


def test_hybrid_dequantized_source_matches_dequantize_then_quantize(cuda):
    """Columnwise-from-dequantized equals: dequantize the rowwise codes to BF16 with
    fp8_dequantize, then cast-transpose that tensor in the columnwise format."""
    x = random_input((256, 256), torch.bfloat16, 43, cuda)
    s_row, s_col = dev_scalar(np.float32(64.0), cuda), dev_scalar(np.float32(2.5), cuda)
    q_row = torch.empty((256, 256), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((256, 256), dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_hybrid(x, E4M3, s_row, q_row, E5M2, s_col, q_col, fq.COLUMNWISE_FROM_ROWWISE_DEQUANTIZED)
    si = dev_scalar(np.float32(1.0 / 64.0), cuda)
    y = torch.empty((256, 256), dtype=torch.bfloat16, device=cuda)
    fq.fp8_dequantize(q_row, E4M3, si, y)
    q2 = torch.empty_like(q_col)
    fq.fp8_quantize_cast_transpose(y, E5M2, s_col, None, q2)
    torch.cuda.synchronize()
    assert torch.equal(q_col, q2)


def test_hybrid_rejects_bad_source(cuda):
    x = torch.zeros((16, 16), dtype=torch.bfloat16, device=cuda)
    s = dev_scalar(np.float32(1.0), cuda)
    q = torch.empty((16, 16), dtype=torch.uint8, device=cuda)
    with pytest.raises(fq.Fp8Error):
        fq.fp8_quantize_hybrid(x, E4M3, s, q, E5M2, s, q.clone(), 7)


# ---------------------------------------------------------------------------
# Back-to-back reductions on one stream
# ---------------------------------------------------------------------------

def test_back_to_back_reductions_do_not_mix(cuda, oracle):
    """A large amax / count followed by a small one on the same stream (and the
    same workspace) must report the small one."""
    big = random_input(3_000_000, torch.bfloat16, 61, cuda) * 1000
    small = random_input(5000, torch.bfloat16, 62, cuda)
    am, s, si = (torch.empty(1, device=cuda) for _ in range(3))
    sat = torch.empty(1, dtype=torch.int64, device=cuda)
    q_big = torch.empty(big.shape, dtype=torch.uint8, device=cuda)
    q_small = torch.empty(small.shape, dtype=torch.uint8, device=cuda)
    one = dev_scalar(np.float32(1.0), cuda)
    for _ in range(2):
        fq.fp8_amax(big, am)
        fq.fp8_amax(small, am, E4M3, 0, s, si)
        torch.cuda.synchronize()
        assert f32_bits(am.item()) == f32_bits(oracle.amax(host_bits(small)))
        fq.fp8_quantize(big, E4M3, one, q_big, am, sat)
        fq.fp8_quantize(small, E4M3, one, q_small, am, sat)
        torch.cuda.synchronize()
        _, wsat = oracle.quantize(host_bits(small), E4M3, np.float32(1.0))
        assert sat.item() == wsat and f32_bits(am.item()) == f32_bits(oracle.amax(host_bits(small)))



@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_cast_transpose_fused_amax_walks_tiles(cuda, oracle, dtype):
    """12416 x 11520 (97 x 90 = 8730 tiles, more than the 8192 partial slots):
    the fused-amax CTAs each take several tiles."""
    g = torch.Generator(device="cpu").manual_seed(64)
    x = (torch.randn((12416, 11520), generator=g) * 3).to(dtype).to(cuda)
    x[12415, 11519] = -640.0  # exact in BF16 and fp32
    s = dev_scalar(np.float32(0.5), cuda)
    q_row = torch.empty((12416, 11520), dtype=torch.uint8, device=cuda)
    q_col = torch.empty((11520, 12416), dtype=torch.uint8, device=cuda)
    am = torch.empty(1, device=cuda)
    fq.fp8_quantize_cast_transpose(x, E4M3, s, q_row, q_col, am)
    torch.cuda.synchronize()
    assert am.item() == 640.0
    xb = host_bits(x)
    wq, _ = oracle.quantize(xb, E4M3, np.float32(0.5), oracle.default_threads())
    assert np.array_equal(q_row.cpu().numpy(), wq)
    assert np.array_equal(q_col.cpu().numpy(), np.ascontiguousarray(wq.T))
