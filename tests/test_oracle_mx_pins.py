"""Pins of the oracle's MXFP8 functions ("Megatron FP8" §10, §16; "Low
Precision Training and Rollout", "MXFP8 (Blackwell only)").  Expected values
come from the pages (tests/golden/mx_overhead.txt), from the E8M0 definition,
from an exhaustive nearest search written here, or from invariants."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from conftest import golden
from test_oracle_pins import brute_force_encode, bf16_values

E4M3, E5M2 = 0, 1
EMAX = {E4M3: 8, E5M2: 15}


def test_e8m0_range_matches_page(oracle):
    # 8 exponent bits, no mantissa, no sign: 2^-127 .. 2^127, one NaN code
    vals = [oracle.e8m0_decode(c) for c in range(256)]
    assert vals[0] == 2.0 ** -127 and vals[254] == 2.0 ** 127 and math.isnan(vals[255])
    assert len(set(vals[:255])) == 255
    assert all(vals[i + 1] == 2 * vals[i] for i in range(254))


def test_mx_overhead_arithmetic(oracle):
    g = golden("mx_overhead.txt")
    n = g["elements"]
    x = np.ones((1, n), dtype=np.float32)
    q, sc = oracle.quantize_mx(x, E4M3)
    assert q.nbytes == n and sc.nbytes == g["scale_bytes"] and q.nbytes + sc.nbytes == g["total_bytes"]
    assert sc.nbytes / q.nbytes == g["overhead"] == 1 / g["block"]
    # 16K x 16K FP8 weight: 256 MB of codes, 8 MB of scales (§10)
    assert 16384 * 16384 / 2 ** 20 == 256 and 16384 * (16384 // 32) / 2 ** 20 == 8


def brute_force_mx(x: np.ndarray, fmt: int):
    """Shared exponent from math.frexp (floor(log2 amax) - emax), codes by exhaustive search."""
    rows, cols = x.shape
    nb = -(-cols // 32)
    q = np.zeros(x.shape, np.uint8)
    sc = np.zeros((rows, nb), np.uint8)
    for r in range(rows):
        for b in range(nb):
            blk = x[r, b * 32:(b + 1) * 32].astype(np.float64)
            if not np.all(np.isfinite(blk)):
                sc[r, b] = 0xFF
                q[r, b * 32:(b + 1) * 32] = 0x7F
                continue
            a = np.abs(blk).max()
            se = -127 if a == 0 else max(-127, min(127, math.frexp(a)[1] - 1 - EMAX[fmt]))
            sc[r, b] = se + 127
            m = np.float32(2.0 ** -se)
            q[r, b * 32:(b + 1) * 32] = brute_force_encode(x[r, b * 32:(b + 1) * 32].astype(np.float32) * m, fmt)
    return q, sc


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx_quantize_small_vs_brute_force(oracle, fmt):
    rng = np.random.default_rng(fmt + 10)
    x = (rng.standard_normal((7, 100)) * np.exp(3 * rng.standard_normal((7, 1)))).astype(np.float32)
    x[0, :32] = 0.0                     # all-zero block -> 2^-127
    x[1, 5] = np.inf                    # non-finite block -> NaN scale
    x[2, 40] = 3e-39                    # subnormal-magnitude block member
    x[3, 64:96] = 1e-38                 # tiny block: exponent clamped at -127
    q, sc = oracle.quantize_mx(x, fmt)
    wq, wsc = brute_force_mx(x, fmt)
    assert np.array_equal(sc, wsc)
    assert np.array_equal(q, wq)
    assert sc[0, 0] == 0 and sc[1, 0] == 0xFF


def test_mx_block_max_lands_in_top_binade_and_pow2_invariance(oracle):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 256)) * 5).astype(np.float32)
    q, sc = oracle.quantize_mx(x, E4M3)
    dec = oracle.decode(q, E4M3)
    for r in range(0, 64, 7):
        for b in range(8):
            blk = np.abs(dec[r, b * 32:(b + 1) * 32])
            assert 256.0 <= blk.max() <= 448.0  # amax / 2^shared_exp lies in [2^8, 2^9), clamped to 448
    for k in (-20, 3):
        q2, sc2 = oracle.quantize_mx(x * np.float32(2.0 ** k), E4M3)
        assert np.array_equal(q2, q) and np.array_equal(sc2.astype(int), sc.astype(int) + k)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qb, scb = oracle.quantize_mx(bits, E4M3)
    wq, wsc = brute_force_mx(bf16_values(bits).reshape(x.shape), E4M3)
    assert np.array_equal(qb, wq) and np.array_equal(scb, wsc)
    qt, sct = oracle.quantize_mx(x, E4M3, threads=3)
    assert np.array_equal(qt, q) and np.array_equal(sct, sc)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx_dequantize_is_decode_times_power_of_two(oracle, fmt):
    rng = np.random.default_rng(8)
    q = rng.integers(0, 256, size=(5, 64), dtype=np.uint8)
    sc = rng.integers(100, 150, size=(5, 2), dtype=np.uint8)
    sc[4, 1] = 0xFF
    y = oracle.dequantize_mx(q, sc, fmt, out_dt=oracle.FP32)
    ref = torch.from_numpy(q).view(torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2).double().numpy()
    want = ref * np.repeat(2.0 ** (sc.astype(np.float64) - 127), 32, axis=1)
    want[4, 32:] = np.nan
    fin = np.isfinite(want)
    assert np.array_equal(y[fin], want[fin].astype(np.float32))
    assert np.array_equal(np.isnan(y), np.isnan(want))


def test_block128_to_mx_rescale_is_lossless(oracle):
    rng = np.random.default_rng(6)
    rows, cols = 256, 384
    # per-128x128-block amax equal to 448 * 2^k so that every block scale is a power of two
    k = rng.integers(-10, 10, size=(2, 3))
    x = np.clip(rng.standard_normal((rows, cols)), -3, 3).astype(np.float32)
    for i in range(2):
        for j in range(3):
            blk = x[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            blk *= np.float32(448.0 * 2.0 ** k[i, j]) / np.abs(blk).max()
            blk[0, 0] = np.float32(448.0 * 2.0 ** k[i, j])
    q, si = oracle.quantize_block(x, 128, 128, E4M3)
    assert np.array_equal(si, (2.0 ** k).astype(np.float32))
    mx, bad = oracle.block128_scales_to_mx(si, rows, cols)
    assert bad == 0 and mx.shape == (rows, cols // 32)
    y_block = oracle.dequantize(q, E4M3, si, 128, 128, out_dt=oracle.FP32)
    y_mx = oracle.dequantize_mx(q, mx, E4M3, out_dt=oracle.FP32)
    assert np.array_equal(y_block, y_mx)
    si2 = si.copy()
    si2[1, 2] = 3.0
    mx2, bad2 = oracle.block128_scales_to_mx(si2, rows, cols)
    assert bad2 == 1 and np.all(mx2[128:, 256 // 32:] == 0xFF) and np.array_equal(mx2[:128], mx[:128])
