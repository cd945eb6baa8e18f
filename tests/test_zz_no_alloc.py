"""fp8_amax_noalloc: the amax + current-scale entry point that allocates no
device memory, for callers that cannot allocate (stream capture in the global
mode, fixed-budget engines and plugins, allocator-owned frameworks).

It must give the same amax, scale and scale_inv as fp8_amax, call after call,
while keeping its scratch in a fixed device array.  This file is collected
last so that a run stopping at the first failure has run everything else."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq

MAX_ELEMS = 1 << 28


def _bits(t):
    return int(t.cpu().numpy().view(np.uint32)[0])


def test_noalloc_rejects_inputs_beyond_its_scratch(native_lib):
    # rejected on the host before any device work (the pointer is never read)
    st = native_lib.fp8_amax_noalloc(0x1000, fq.DT_BF16, MAX_ELEMS + 1, 0x2000, 0, 0, None, None, None)
    assert st == 2
    assert "exceeds the fixed scratch capacity" in native_lib.fp8_last_error_message().decode()


@pytest.mark.gpu
def test_noalloc_matches_allocating_amax_two_calls_in_a_row(cuda):
    g = torch.Generator(device="cpu").manual_seed(1234)
    cases = [
        (torch.bfloat16, 0, fq.E4M3, 0),
        (torch.bfloat16, 1, fq.E4M3, 0),
        (torch.bfloat16, 65537, fq.E5M2, 1),
        (torch.float32, 300_001, fq.E4M3, 3),
        (torch.bfloat16, 8192 * 8192, fq.E5M2, 0),
    ]
    xs = []
    for dtype, n, fmt, margin in cases:
        x = (torch.randn(n, generator=g) * torch.exp(2 * torch.randn(n, generator=g))).to(dtype).to(cuda)
        xs.append((x, fmt, margin))
    base = torch.randn(4099, generator=g).to(torch.bfloat16).to(cuda)
    xs.append((base[3:], fq.E4M3, 0))  # not 16-byte aligned
    nan = torch.randn(100_000, generator=g).to(torch.bfloat16).to(cuda)
    nan[777] = float("nan")
    xs.append((nan, fq.E4M3, 0))
    for call in range(2):  # two calls in a row share (and reuse) the fixed scratch
        for x, fmt, margin in xs:
            out = [torch.full((1,), -1.0, device=cuda) for _ in range(6)]
            fq.fp8_amax(x, out[0], fmt, margin, out[1], out[2])
            fq.fp8_amax_noalloc(x, out[3], fmt, margin, out[4], out[5])
            torch.cuda.synchronize()
            ref, got = [_bits(t) for t in out[:3]], [_bits(t) for t in out[3:]]
            assert got == ref, (call, x.numel(), x.dtype)


@pytest.mark.gpu
def test_noalloc_at_its_capacity(cuda):
    """2^28 BF16 elements (every one of the 4096 scratch slots in use) with the
    maximum in the last element, and 2^28 - 1 elements starting one element
    past a 16-byte boundary (the element-at-a-time path), each against
    fp8_amax bit for bit, two calls in a row."""
    g = torch.Generator(device=cuda).manual_seed(4321)
    full = torch.randn(MAX_ELEMS, generator=g, device=cuda).to(torch.bfloat16)
    full[-1] = -1024.0  # above every N(0, 1) draw: the last CTA's slot holds the maximum
    cases = [(full, fq.E4M3, 0), (full[1:], fq.E5M2, 2)]
    for call in range(2):
        for x, fmt, margin in cases:
            out = [torch.full((1,), -1.0, device=cuda) for _ in range(6)]
            fq.fp8_amax(x, out[0], fmt, margin, out[1], out[2])
            fq.fp8_amax_noalloc(x, out[3], fmt, margin, out[4], out[5])
            torch.cuda.synchronize()
            ref, got = [_bits(t) for t in out[:3]], [_bits(t) for t in out[3:]]
            assert got == ref, (call, x.numel())
            assert out[3].item() == 1024.0
