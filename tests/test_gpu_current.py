"""Current scaling in one call (fp8_quantize_current) against the oracle.

"Megatron FP8" §10 (the scale of a current-scaling cast comes from the amax
of the tensor being cast) and §4 (amax -> scale with margin -> cast).  The
call must give exactly what fp8_amax followed by fp8_quantize gives.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq

from test_gpu_parity import f32_bits, host_bits, random_input, with_specials

pytestmark = pytest.mark.gpu
E4M3, E5M2 = fq.E4M3, fq.E5M2


def run_current(x, fmt, margin):
    dev = x.device
    q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    am, s, si = (torch.full((1,), -5.0, device=dev) for _ in range(3))
    fq.fp8_quantize_current(x, fmt, q, margin, am, s, si)
    torch.cuda.synchronize()
    return q, am.item(), s.item(), si.item()


def check_against_oracle(oracle, x, fmt, margin):
    q, am, s, si = run_current(x, fmt, margin)
    xb = host_bits(x)
    want_amax = oracle.amax(xb)
    ws, wsi = oracle.compute_scale(want_amax, fmt, margin)
    assert f32_bits(am) == f32_bits(want_amax)
    assert (f32_bits(s), f32_bits(si)) == (f32_bits(ws), f32_bits(wsi))
    wq, _ = oracle.quantize(xb, fmt, ws)
    assert np.array_equal(q.cpu().numpy(), wq)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("n", [1, 7, 15, 16, 17, 1000, 16385, (1 << 20) + 3, 3_000_001])
def test_current_matches_oracle(cuda, oracle, dtype, fmt, n):
    check_against_oracle(oracle, random_input(n, dtype, 300 + n, cuda), fmt, 1)


@pytest.mark.parametrize("margin", [-1, 0, 3])
def test_current_margins_and_specials(cuda, oracle, margin):
    x = random_input(2_000_003, torch.bfloat16, 12, cuda)
    check_against_oracle(oracle, x, E5M2, margin)
    x[77] = float("inf")  # amax Inf -> scale 1
    check_against_oracle(oracle, x, E4M3, margin)
    check_against_oracle(oracle, with_specials(x.clone(), 4), E4M3, margin)  # NaN -> canonical amax


def test_current_zero_empty_and_unaligned(cuda, oracle):
    q, am, s, si = run_current(torch.zeros(4099, dtype=torch.bfloat16, device=cuda), E4M3, 0)
    assert (am, s, si) == (0.0, 1.0, 1.0) and int(q.sum()) == 0
    q, am, s, si = run_current(torch.zeros(0, dtype=torch.bfloat16, device=cuda), E4M3, 0)
    assert (am, s, si) == (0.0, 1.0, 1.0)
    base = random_input(300_001, torch.bfloat16, 15, cuda)
    check_against_oracle(oracle, base[3:], E4M3, 0)  # unaligned: the fp8_amax + fp8_quantize kernels
    q = torch.empty(1000, dtype=torch.uint8, device=cuda)
    fq.fp8_quantize_current(base[:1000], E4M3, q)  # no scalar outputs requested
    torch.cuda.synchronize()
    ws, _ = oracle.compute_scale(oracle.amax(host_bits(base[:1000])), E4M3, 0)
    assert np.array_equal(q.cpu().numpy(), oracle.quantize(host_bits(base[:1000]), E4M3, ws)[0])


def test_current_equals_amax_then_quantize_full_size(cuda, oracle):
    """8192 x 8192 BF16 (the E5M2 gradient size): identical to fp8_amax + fp8_quantize,
    and sampled codes equal the oracle's."""
    g = torch.Generator(device=cuda).manual_seed(21)
    x = (torch.randn((8192, 8192), generator=g, device=cuda) * 3e-3).to(torch.bfloat16)
    q, am, s, si = run_current(x, E5M2, 0)
    am2, s2, si2 = (torch.empty(1, device=cuda) for _ in range(3))
    fq.fp8_amax(x, am2, E5M2, 0, s2, si2)
    q2 = torch.empty_like(q)
    fq.fp8_quantize(x, E5M2, s2, q2)
    torch.cuda.synchronize()
    assert (f32_bits(am), f32_bits(s), f32_bits(si)) == (f32_bits(am2.item()), f32_bits(s2.item()),
                                                         f32_bits(si2.item()))
    assert torch.equal(q, q2)
    idx = torch.randint(0, x.numel(), (200_000,), generator=g, device=cuda)
    wq, _ = oracle.quantize(host_bits(x.view(-1)[idx]), E5M2, np.float32(s))
    assert np.array_equal(q.view(-1)[idx].cpu().numpy(), wq)


def test_current_in_a_captured_graph(cuda, oracle):
    xs = [random_input(1_000_000 + 16 * i, torch.bfloat16, 40 + i, cuda) for i in range(3)]
    qs = [torch.empty(x.shape, dtype=torch.uint8, device=cuda) for x in xs]
    ss = [torch.empty(1, device=cuda) for _ in xs]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for x, q, s in zip(xs, qs, ss):
            fq.fp8_quantize_current(x, E4M3, q, 0, None, s, None)
    for x in xs:
        x.mul_(3.0)
    graph.replay()
    torch.cuda.synchronize()
    for x, q, s in zip(xs, qs, ss):
        ws, _ = oracle.compute_scale(oracle.amax(host_bits(x)), E4M3, 0)
        assert f32_bits(s.item()) == f32_bits(ws)
        assert np.array_equal(q.cpu().numpy(), oracle.quantize(host_bits(x), E4M3, ws)[0])


@pytest.mark.parametrize("dtype,n", [(torch.bfloat16, 7_000_003), (torch.float32, 3_200_001)])
def test_current_above_the_cast_reduction_threshold(cuda, oracle, dtype, n):
    """Just above 256 amax partials the call switches to amax + finalize + cast."""
    check_against_oracle(oracle, random_input(n, dtype, 90, cuda), E4M3, 1)


@pytest.mark.parametrize("dtype,n", [
    (torch.bfloat16, 8), (torch.bfloat16, 65536 - 1), (torch.bfloat16, 65536), (torch.bfloat16, 65537),
    (torch.bfloat16, 3 * 65536 + 5), (torch.bfloat16, 9 * 65536 + 3), (torch.bfloat16, (1 << 20) - 7),
    (torch.bfloat16, 1 << 20), (torch.bfloat16, (1 << 20) + 1),
    (torch.float32, 4), (torch.float32, 32768 + 1), (torch.float32, 5 * 32768 + 2), (torch.float32, 1 << 19),
    (torch.float32, (1 << 19) + 3)])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_current_small_tensor_sizes(cuda, oracle, dtype, fmt, n):
    """Small tensors: sizes around whole chunks of the amax kernel and of the
    cast, 2 MiB, and ragged tails, with special values planted."""
    x = with_specials(random_input(n, dtype, 500 + n, cuda), n)
    check_against_oracle(oracle, x, fmt, 0)
    check_against_oracle(oracle, random_input(n, dtype, 600 + n, cuda), fmt, 2)


def test_current_planted_maximum_positions(cuda, oracle):
    """The amax sits in the ragged tail, in the last chunk and in an inner chunk."""
    for pos in (1048574, 1048555, 948575):
        x = random_input(1048575, torch.bfloat16, 77, cuda, spread=False)  # |x| < 1000
        x[pos] = -32768.0  # exact in BF16
        q, am, s, si = run_current(x, E4M3, 0)
        assert am == 32768.0
        check_against_oracle(oracle, x, E4M3, 0)
