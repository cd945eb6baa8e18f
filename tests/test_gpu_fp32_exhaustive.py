"""Exhaustive FP32-input parity: all 2^32 fp32 bit patterns through fp8_quantize.

"Megatron FP8" §4 defines the cast as one fp32 multiply x * scale followed by
a clamp to +-FP8_MAX; §2 fixes the formats (E4M3FN saturates to +-448 and has
no Inf, E5M2 keeps +-Inf).  FP32 inputs reach round-to-nearest ties, subnormal
products and the saturation bands (448..464 for E4M3, 57344..61440 for E5M2)
in ways that BF16 inputs never do, and the library converts them on a path of
their own (four fp32 values per 16-byte load, with an element-exact fixup).

For both formats, at scale 1 and at the non-power-of-two scale fl32(448/1000),
every pattern goes through three kernel variants:
  * the cast with fused amax and saturation count (16-byte path, fixups taken
    whenever a chunk saturates),
  * the plain cast (16-byte path, saturation left to the hardware conversion),
  * the element-at-a-time path (input and output one element off a 16-byte
    boundary).
Each is compared bit for bit with the oracle's codes, and the count and amax
with the oracle's, in chunks of 2^28 patterns (1 GiB of input on the device).
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28
SCALES = (np.float32(1.0), np.float32(448.0) / np.float32(1000.0))


def test_all_fp32_patterns(cuda, oracle):
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    x_dev = torch.empty(CHUNK, dtype=torch.float32, device=cuda)
    q_dev = torch.empty(CHUNK, dtype=torch.uint8, device=cuda)
    q2_dev = torch.empty(CHUNK, dtype=torch.uint8, device=cuda)
    q3_dev = torch.empty(CHUNK, dtype=torch.uint8, device=cuda)
    amax_dev = torch.empty(1, dtype=torch.float32, device=cuda)
    sat_dev = torch.empty(1, dtype=torch.int64, device=cuda)
    scale_dev = {float(s): torch.tensor([s], dtype=torch.float32, device=cuda) for s in SCALES}
    total_sat = {}
    for c in range(1 << 32 >> 28):
        xh = np.arange(c * CHUNK, (c + 1) * CHUNK, dtype=np.uint32).view(np.float32)
        x_dev.copy_(torch.from_numpy(xh))
        want_amax = oracle.amax(xh, threads)
        for fmt in (fq.E4M3, fq.E5M2):
            for s in SCALES:
                sd = scale_dev[float(s)]
                fq.fp8_quantize(x_dev, fmt, sd, q_dev, amax_dev, sat_dev)
                fq.fp8_quantize(x_dev, fmt, sd, q2_dev)
                fq.fp8_quantize(x_dev[1:], fmt, sd, q3_dev[1:])
                want_q, want_sat = oracle.quantize(xh, fmt, s, threads)
                where = f"chunk {c:#x}, fmt {fmt}, scale {float(s)!r}"
                got = q_dev.cpu().numpy()
                assert np.array_equal(got, want_q), f"{where}: fused amax + count cast, first bad pattern " \
                    f"{int(np.flatnonzero(got != want_q)[0]) + c * CHUNK:#010x}"
                got = q2_dev.cpu().numpy()
                assert np.array_equal(got, want_q), f"{where}: plain cast, first bad pattern " \
                    f"{int(np.flatnonzero(got != want_q)[0]) + c * CHUNK:#010x}"
                got = q3_dev[1:].cpu().numpy()
                assert np.array_equal(got, want_q[1:]), f"{where}: element path, first bad pattern " \
                    f"{int(np.flatnonzero(got != want_q[1:])[0]) + 1 + c * CHUNK:#010x}"
                assert int(sat_dev.item()) == want_sat, where
                assert amax_dev.cpu().numpy().view(np.uint32)[0] == np.float32(want_amax).view(np.uint32), where
                key = (fmt, float(s))
                total_sat[key] = total_sat.get(key, 0) + want_sat
    # Closed forms of the counts over all patterns: a finite x saturates when
    # |fl32(x * s)| > FP8_MAX, so at scale 1 the count is the number of finite
    # fp32 magnitudes above FP8_MAX, times two signs.
    for fmt, fmax in ((fq.E4M3, 448.0), (fq.E5M2, 57344.0)):
        above = 0x7F800000 - (int(np.float32(fmax).view(np.uint32)) + 1)
        assert total_sat[(fmt, 1.0)] == 2 * above, fmt
    print(f"all 2^32 fp32 patterns x 2 formats x 2 scales x 3 variants: {time.perf_counter() - t0:.1f} s")
