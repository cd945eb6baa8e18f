"""Grouped current scaling (fp8_amax_grouped + fp8_quantize_grouped) against the
oracle and against the per-tensor entry points.

"Megatron FP8" §21: each expert of an MoE layer keeps its own per-tensor
scaling state; the grouped calls compute every tensor's amax, current scale
and codes in one kernel launch each (plus one finalize for the amax).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq

from test_gpu_parity import f32_bits, host_bits, random_input, with_specials

pytestmark = pytest.mark.gpu
E4M3, E5M2 = fq.E4M3, fq.E5M2

SIZES = [0, 1, 15, 16, 17, 1000, 16384, 16385, 70_001, 300_000]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_grouped_matches_oracle(cuda, oracle, dtype, fmt):
    xs = []
    for i, n in enumerate(SIZES):
        x = random_input(n, dtype, 500 + i, cuda)
        if i == 8:
            x = with_specials(x, 9)  # one tensor with Inf / NaN: amax NaN, scale 1
        xs.append(x)
    m = len(xs)
    am, s, si = (torch.full((m,), -3.0, device=cuda) for _ in range(3))
    fq.fp8_amax_grouped(xs, am, fmt, 1, s, si)
    qs = [torch.empty(x.shape, dtype=torch.uint8, device=cuda) for x in xs]
    fq.fp8_quantize_grouped(xs, fmt, s, qs)
    torch.cuda.synchronize()
    for i, x in enumerate(xs):
        xb = host_bits(x)
        wa = oracle.amax(xb)
        ws, wsi = oracle.compute_scale(wa, fmt, 1)
        assert f32_bits(am[i].item()) == f32_bits(wa), i
        assert (f32_bits(s[i].item()), f32_bits(si[i].item())) == (f32_bits(ws), f32_bits(wsi)), i
        wq, _ = oracle.quantize(xb, fmt, ws)
        assert np.array_equal(qs[i].cpu().numpy(), wq), i


def test_grouped_matches_per_tensor_calls(cuda):
    """32 expert-sized tensors (about 500M elements: the amax CTAs then cover
    several chunks each) against fp8_amax + fp8_quantize per tensor."""
    g = torch.Generator(device=cuda).manual_seed(5)
    rows = torch.randint(256, 4096, (32,), generator=g, device=cuda).tolist()
    xs = [(torch.randn((int(r), 7168), generator=g, device=cuda) * (i + 1)).to(torch.bfloat16)
          for i, r in enumerate(rows)]
    m = len(xs)
    am, s, si = (torch.empty(m, device=cuda) for _ in range(3))
    fq.fp8_amax_grouped(xs, am, E4M3, 0, s, si)
    qs = [torch.empty(x.shape, dtype=torch.uint8, device=cuda) for x in xs]
    fq.fp8_quantize_grouped(xs, E4M3, s, qs)
    a1, s1, si1 = (torch.empty(1, device=cuda) for _ in range(3))
    for i, x in enumerate(xs):
        fq.fp8_amax(x, a1, E4M3, 0, s1, si1)
        q1 = torch.empty_like(qs[i])
        fq.fp8_quantize(x, E4M3, s1, q1)
        torch.cuda.synchronize()
        assert f32_bits(am[i].item()) == f32_bits(a1.item()) and f32_bits(s[i].item()) == f32_bits(s1.item()), i
        assert torch.equal(qs[i], q1), i


def test_grouped_at_the_128_tensor_limit(cuda, oracle):
    """The largest group a table takes: 128 tensors of mixed sizes (empty ones
    included), E5M2, margin 2."""
    sizes = [(i * 977) % 6001 for i in range(128)]
    xs = [random_input(n, torch.bfloat16, 900 + i, cuda) for i, n in enumerate(sizes)]
    am, s, si = (torch.full((128,), -3.0, device=cuda) for _ in range(3))
    fq.fp8_amax_grouped(xs, am, E5M2, 2, s, si)
    qs = [torch.empty(x.shape, dtype=torch.uint8, device=cuda) for x in xs]
    fq.fp8_quantize_grouped(xs, E5M2, s, qs)
    torch.cuda.synchronize()
    for i, x in enumerate(xs):
        xb = host_bits(x)
        wa = oracle.amax(xb)
        ws, wsi = oracle.compute_scale(wa, E5M2, 2)
        assert f32_bits(am[i].item()) == f32_bits(wa), i
        assert (f32_bits(s[i].item()), f32_bits(si[i].item())) == (f32_bits(ws), f32_bits(wsi)), i
        wq, _ = oracle.quantize(xb, E5M2, ws)
        assert np.array_equal(qs[i].cpu().numpy(), wq), i


def test_grouped_all_empty(cuda):
    """A group of empty tensors: amax 0, scale and scale_inv 1, nothing written."""
    xs = [torch.empty(0, dtype=torch.bfloat16, device=cuda) for _ in range(5)]
    am, s, si = (torch.full((5,), -3.0, device=cuda) for _ in range(3))
    fq.fp8_amax_grouped(xs, am, E4M3, 0, s, si)
    fq.fp8_quantize_grouped(xs, E4M3, s, [torch.empty(0, dtype=torch.uint8, device=cuda) for _ in range(5)])
    torch.cuda.synchronize()
    assert am.tolist() == [0.0] * 5 and s.tolist() == [1.0] * 5 and si.tolist() == [1.0] * 5


def test_grouped_rejects_bad_tables(cuda):
    base = torch.zeros(1000, dtype=torch.bfloat16, device=cuda)
    am = torch.empty(2, device=cuda)
    with pytest.raises(fq.Fp8Error) as e:
        fq.fp8_amax_grouped([base[:64], base[1:65]], am)  # second tensor not 16-byte aligned
    assert e.value.status == 2
    with pytest.raises(fq.Fp8Error) as e:
        fq.fp8_amax_grouped([base[:8]] * 129, torch.empty(129, device=cuda))
    assert e.value.status == 1
    with pytest.raises(ValueError):
        fq.fp8_amax_grouped([base[:8]] * 3, am)  # outputs shorter than the group
