"""Pins of the CPU oracle to facts the pages and the mathematics fix.

Nothing here compares the oracle with itself: every expected value comes from
a page (tests/golden, each fixture citing its section), a closed form, an
independent brute-force search written in this file, or a library routine
(torch's float8 dtypes, numpy).  A dropped term, a wrong sign, a wrong index
or a transposed operand in the oracle fails at least one test below.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from conftest import golden

E4M3, E5M2 = 0, 1
MANT = {E4M3: 3, E5M2: 2}
EXPB = {E4M3: 4, E5M2: 5}
TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ grids

def grid_from_fields(exp_bits: int, mant_bits: int, fn: bool) -> list[float]:
    """Non-negative finite values of a (1, exp_bits, mant_bits) format, built
    from the field definitions of "Megatron FP8" §2/§3: bias 2^(k-1)-1,
    subnormals m * 2^(1-bias-M), normals (1 + m/2^M) * 2^(e-bias).  The
    all-ones exponent is skipped entirely for IEEE-style formats; for the FN
    variant only its all-ones mantissa (the NaN) is skipped."""
    bias = 2 ** (exp_bits - 1) - 1
    top = 2 ** exp_bits - 1
    vals = set()
    for e in range(top + 1):
        for m in range(2 ** mant_bits):
            if e == top and (not fn or m == 2 ** mant_bits - 1):
                continue
            if e == 0:
                vals.add(math.ldexp(m, 1 - bias - mant_bits))
            else:
                vals.add(math.ldexp(2 ** mant_bits + m, e - bias - mant_bits))
    return sorted(vals)


def brute_force_encode(values: np.ndarray, fmt: int) -> np.ndarray:
    """Nearest finite grid value by exhaustive search over all 256 codes
    (ties to the code with an even mantissa), saturation beyond the largest
    finite value, the sign copied (so -0 and tiny negatives give 0x80), NaN ->
    0x7F, +-Inf -> E5M2 Inf code / E4M3FN max code.  Written without the
    oracle: the code table is torch's float8 decode."""
    codes = np.arange(256, dtype=np.uint8)
    dec = torch.from_numpy(codes).view(TORCH_FP8[fmt]).to(torch.float64).numpy()
    pos = (codes < 0x80) & np.isfinite(dec)
    pcodes, pvals = codes[pos], dec[pos]
    v = np.asarray(values, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    out = np.zeros(v.shape, dtype=np.uint8)
    fin = np.isfinite(v)
    top = pvals.max()
    inside = fin & (a < top)  # at or beyond the largest finite value: saturate
    d = np.abs(a[inside][:, None] - pvals[None, :])  # exact: |a| < 57344 here
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among equidistant neighbours prefer the even code (mantissa LSB 0)
    even = (pcodes & 1) == 0
    pick = np.where(cand & even[None, :], 1, 0) * 2 + cand
    idx = pick.argmax(axis=1)
    out[inside] = pcodes[idx]
    out[fin & (a >= top)] = pcodes[pvals.argmax()]
    sign = (np.signbit(v) & ~np.isnan(v)).astype(np.uint8) << 7
    out = out | np.where(fin, sign, 0).astype(np.uint8)
    inf = np.isinf(v)
    inf_code = 0x7C if fmt == E5M2 else 0x7E
    out[inf] = inf_code | sign[inf]
    out[np.isnan(v)] = 0x7F
    return out


# ---------------------------------------------------------------- formats

@pytest.mark.parametrize("fmt,key", [(E4M3, "e4m3"), (E5M2, "e5m2")])
def test_format_stats_match_page(oracle, fmt, key):
    g = golden("format_stats.txt")
    bias, e_max, mx = oracle.format_stats(fmt)
    assert (bias, e_max, mx) == (g[f"{key}.bias"], g[f"{key}.e_max"], g[f"{key}.max_finite"])
    assert oracle.min_normal(fmt) == g[f"{key}.min_normal"]
    # (2 - 2^-M) * 2^e_max from the same section
    assert mx == (2 - 2.0 ** -MANT[fmt]) * 2.0 ** e_max or fmt == E4M3
    if fmt == E4M3:  # FN: the top binade stops one step short: 1.75 * 2^8
        assert mx == 1.75 * 2.0 ** 8


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decoded_set_equals_enumerated_grid(oracle, fmt):
    dec = oracle.decode(np.arange(256, dtype=np.uint8), fmt).astype(np.float64)
    finite_nonneg = sorted(set(float(v) for v in np.abs(dec[np.isfinite(dec)])))
    grid = grid_from_fields(EXPB[fmt], MANT[fmt], fn=(fmt == E4M3))
    assert finite_nonneg == grid
    assert len(grid) == (127 if fmt == E4M3 else 124)
    assert grid[-1] == (448.0 if fmt == E4M3 else 57344.0)


def test_ieee_style_enumeration_is_not_e4m3fn():
    # The unamended IEEE-style enumeration of (4, 3) stops at 240 with 120
    # values; E4M3FN keeps the all-ones exponent (256 .. 448).  This records
    # the reading that the page's E4M3 is E4M3FN (max 448, §2).
    ieee = grid_from_fields(4, 3, fn=False)
    assert len(ieee) == 120 and ieee[-1] == 240.0
    assert grid_from_fields(4, 3, fn=True)[-8:] == [240.0, 256.0, 288.0, 320.0, 352.0, 384.0, 416.0, 448.0]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_special_codes_and_sign_symmetry(oracle, fmt):
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.decode(codes, fmt)
    nan = set(codes[np.isnan(dec)].tolist())
    inf = set(codes[np.isinf(dec)].tolist())
    if fmt == E4M3:
        assert nan == {0x7F, 0xFF} and inf == set()
    else:
        assert nan == {0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF} and inf == {0x7C, 0xFC}
        assert dec[0x7C] == np.inf and dec[0xFC] == -np.inf
    ok = ~np.isnan(dec)
    flipped = oracle.decode(codes ^ 0x80, fmt)
    assert np.array_equal(flipped[ok], -dec[ok])
    assert np.signbit(dec[0x80]) and dec[0x80] == 0.0


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_matches_torch_float8(oracle, fmt):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(TORCH_FP8[fmt]).float().numpy()
    got = oracle.decode(codes, fmt)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


# ---------------------------------------------------------------- encoding

@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_all_bf16_patterns_at_scale_one_vs_brute_force(oracle, fmt):
    x = bf16_values(ALL_BF16)
    want = brute_force_encode(x, fmt)
    got, _ = oracle.quantize(ALL_BF16, fmt, 1.0)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(ALL_BF16[i]), float(x[i]), hex(got[i]), hex(want[i])) for i in bad[:8]]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("scale", [1.0, 0.2240000069141388, 3.0517578125e-05, 7.0, 1234.5])
def test_scaled_encode_matches_torch_on_finite(oracle, fmt, scale):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 65536, size=200_000, dtype=np.uint32).astype(np.uint16)
    x = bf16_values(bits)
    fin = np.isfinite(x)
    bits, x = bits[fin], x[fin]
    p = x * np.float32(scale)  # IEEE fp32 multiply
    mx = 448.0 if fmt == E4M3 else 57344.0
    want = torch.from_numpy(np.clip(p, -mx, mx)).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    got, _ = oracle.quantize(bits, fmt, scale)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_relative_error_bound(oracle, fmt):
    g = golden("error_bounds.txt")
    key = "e4m3" if fmt == E4M3 else "e5m2"
    bound = g[f"{key}.max_rel_error"]
    assert bound == 2.0 ** -(g[f"{key}.mantissa_bits"] + 1)
    x = bf16_values(ALL_BF16).astype(np.float64)
    lo, hi = oracle.min_normal(fmt), oracle.max_finite(fmt)
    sel = np.isfinite(x) & (np.abs(x) >= lo) & (np.abs(x) <= hi)
    q, _ = oracle.quantize(ALL_BF16[sel], fmt, 1.0)
    back = oracle.decode(q, fmt).astype(np.float64)
    rel = np.abs(back - x[sel]) / np.abs(x[sel])
    assert rel.max() <= bound
    assert rel.max() > bound / 2  # the bound is nearly reached (it is tight)


def test_signed_zero_and_tiny_negatives(oracle):
    for fmt in (E4M3, E5M2):
        assert oracle.quantize_element(-0.0, 1.0, fmt)[0] == 0x80
        assert oracle.quantize_element(-1e-30, 1.0, fmt)[0] == 0x80
        assert oracle.quantize_element(1e-30, 1.0, fmt)[0] == 0x00


def test_special_inputs(oracle):
    inf, nan = float("inf"), float("nan")
    assert oracle.quantize_element(inf, 1.0, E5M2) == (0x7C, 0)
    assert oracle.quantize_element(-inf, 1.0, E5M2) == (0xFC, 0)
    assert oracle.quantize_element(inf, 1.0, E4M3) == (0x7E, 0)
    assert oracle.quantize_element(-inf, 1.0, E4M3) == (0xFE, 0)
    assert oracle.quantize_element(nan, 1.0, E4M3) == (0x7F, 0)
    assert oracle.quantize_element(nan, 1.0, E5M2) == (0x7F, 0)
    # a finite x whose fp32 product overflows saturates (and counts)
    assert oracle.quantize_element(3e38, 10.0, E5M2) == (0x7B, 1)
    assert oracle.quantize_element(-3e38, 10.0, E4M3) == (0xFE, 1)


# ------------------------------------------------------------------ scaling

def test_worked_example_from_page(oracle):
    g = golden("worked_example_scale.txt")
    x = np.array(g["x"], dtype=np.float32)
    fp8_max, margin = np.float32(g["fp8_max"]), g["margin"]
    # the page's formula, in fp32
    amax_p = np.abs(x).max()
    s_star = amax_p / fp8_max
    s = s_star * np.float32(2.0 ** margin)
    clipped = np.clip(x / s, -fp8_max, fp8_max)
    # the oracle (multiplier convention)
    amax = oracle.amax(x)
    scale, scale_inv = oracle.compute_scale(amax, E4M3, margin)
    assert amax == amax_p == np.float32(920.0)
    assert scale_inv == s  # 1 / (448/920 * 2^-1) rounds to exactly the page's s
    assert scale == np.float32(fp8_max / amax_p) * np.float32(0.5)
    mult = x * scale
    ulps = np.abs(mult.view(np.int32) - clipped.view(np.int32))
    assert ulps.max() <= 1 and np.all(np.abs(mult) <= fp8_max)
    q, sat = oracle.quantize(x, E4M3, scale)
    assert sat == 0
    assert list(oracle.decode(q, E4M3)) == [-224.0, 0.875, 128.0]
    assert list(brute_force_encode(clipped, E4M3)) == list(q)


def test_scale_rule_closed_forms(oracle):
    for k in range(-20, 21):
        amax = np.float32(448.0 * 2.0 ** -k)
        s, si = oracle.compute_scale(amax, E4M3, 0)
        assert s == np.float32(2.0 ** k) and si == np.float32(2.0 ** -k)
    for m in range(0, 6):
        s0, _ = oracle.compute_scale(np.float32(3.5), E5M2, 0)
        sm, sim = oracle.compute_scale(np.float32(3.5), E5M2, m)
        assert sm == s0 * np.float32(2.0 ** -m)
        assert sim == np.float32(1.0) / sm
    assert oracle.compute_scale(np.float32(3.5), E4M3, 0)[0] == np.float32(128.0)
    for bad in (0.0, -1.0, np.inf, np.nan):
        assert oracle.compute_scale(bad, E4M3, 0) == (1.0, 1.0)
    s, si = oracle.compute_scale(np.float32(1e-40), E4M3, 0)  # 448/1e-40 overflows fp32
    assert s == np.finfo(np.float32).max and si == np.float32(1.0) / s
    s, si = oracle.compute_scale(np.float32(3e38), E4M3, 126)  # underflows below FLT_MIN
    assert s == np.finfo(np.float32).tiny and si == np.float32(2.0 ** 126)


def test_amax_against_numpy_and_special_cases(oracle):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100_003) * 50).astype(np.float32)
    assert oracle.amax(x) == np.abs(x).max()
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert oracle.amax(bits) == np.abs(bf16_values(bits)).max()
    assert oracle.amax(bits, threads=4) == oracle.amax(bits)
    assert oracle.amax(np.zeros(0, dtype=np.float32)) == 0.0
    y = x.copy()
    y[777] = np.nan
    a = oracle.amax(y)
    assert np.isnan(a) and a.view(np.uint32) == 0x7FC00000
    y = x.copy()
    y[5] = -np.inf
    assert oracle.amax(y) == np.inf


def test_saturation_count_by_construction(oracle):
    rng = np.random.default_rng(11)
    n, k = 50_000, 37
    x = rng.uniform(-100, 100, n).astype(np.float32)
    scale = np.float32(2.0)  # |x * scale| <= 200 < 448: nothing saturates
    idx = rng.choice(n, k, replace=False)
    x[idx] = np.where(rng.random(k) < 0.5, -1.0, 1.0) * rng.uniform(225, 1e6, k)  # > 448 after scaling
    x[rng.choice(np.setdiff1d(np.arange(n), idx), 3, replace=False)] = np.inf  # Inf is not counted
    q, sat = oracle.quantize(x, E4M3, scale)
    assert sat == k
    q, sat = oracle.quantize(x, E4M3, scale, threads=3)
    assert sat == k
    # exactly FP8_MAX after scaling is not saturated
    assert oracle.quantize(np.array([224.0], np.float32), E4M3, 2.0)[1] == 0


# ---------------------------------------------------------- delayed scaling

def test_delayed_zero_history_gives_scale_one(oracle):
    g = golden("delayed_recipe.txt")
    h = np.zeros(g["history_len"], dtype=np.float32)
    assert oracle.update_delayed(h, 0, None, oracle.ALGO_MAX, E4M3, 0) == (g["scale_when_history_zero"],) * 2


def test_delayed_window_semantics(oracle):
    rng = np.random.default_rng(5)
    amaxes = (rng.random(40) * 100).astype(np.float32)
    L = 4
    h = np.zeros(L, dtype=np.float32)
    for k, a in enumerate(amaxes):
        s, si = oracle.update_delayed(h, k, a, oracle.ALGO_MAX, E4M3, 0)
        window = amaxes[max(0, k - L + 1): k + 1]  # the last L recorded amaxes, this one included
        assert s == np.float32(448.0) / window.max()
        assert h[k % L] == a
        s2, _ = oracle.update_delayed(h.copy(), k, None, oracle.ALGO_MOST_RECENT, E4M3, 0)
        assert s2 == np.float32(448.0) / a


def test_delayed_history_one_most_recent_equals_current(oracle):
    rng = np.random.default_rng(9)
    for margin in (0, 1, 3):
        for fmt in (E4M3, E5M2):
            a = np.float32(rng.random() * 1e3)
            h = np.zeros(1, dtype=np.float32)
            assert oracle.update_delayed(h, 17, a, oracle.ALGO_MOST_RECENT, fmt, margin) == \
                oracle.compute_scale(a, fmt, margin)


def test_delayed_nan_in_history(oracle):
    h = np.array([1.0, np.nan, 3.0], dtype=np.float32)
    assert oracle.update_delayed(h, 0, None, oracle.ALGO_MAX, E4M3, 0) == (1.0, 1.0)


# --------------------------------------------------------- cast-transpose

def test_cast_transpose_is_transpose_of_rowwise(oracle):
    rng = np.random.default_rng(1)
    x = torch.from_numpy((rng.standard_normal((37, 53)) * 30).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    scale = np.float32(3.25)
    q_row, q_col = oracle.cast_transpose(bits, E4M3, scale)
    flat, _ = oracle.quantize(bits.ravel(), E4M3, scale)
    assert np.array_equal(q_row.ravel(), flat)
    assert q_col.shape == (53, 37)
    assert np.array_equal(q_col, q_row.T)
    assert np.array_equal(q_row, brute_force_encode(bf16_values(bits) * scale, E4M3))
    r2, c2 = oracle.cast_transpose(bits, E4M3, scale, threads=3)
    assert np.array_equal(r2, q_row) and np.array_equal(c2, q_col)


# --------------------------------------------------------------- blockwise

def brute_force_block(x: np.ndarray, br: int, bc: int, fmt: int):
    """Per-block amax with numpy, the scale from the §4 multiplier form in
    fp32, codes by exhaustive nearest search."""
    rows, cols = x.shape
    mx = np.float32(448.0 if fmt == E4M3 else 57344.0)
    nbr, nbc = -(-rows // br), -(-cols // bc)
    q = np.zeros(x.shape, np.uint8)
    si = np.zeros((nbr, nbc), np.float32)
    for i in range(nbr):
        for j in range(nbc):
            blk = x[i * br:(i + 1) * br, j * bc:(j + 1) * bc]
            a = np.abs(blk).max()
            s = mx / a if a > 0 else np.float32(1.0)
            si[i, j] = np.float32(1.0) / s
            q[i * br:(i + 1) * br, j * bc:(j + 1) * bc] = brute_force_encode(blk * s, fmt)
    return q, si


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("br,bc", [(2, 3), (1, 4), (4, 4)])
def test_block_quantize_small_blocks_vs_brute_force(oracle, fmt, br, bc):
    rng = np.random.default_rng(br * 10 + bc)
    x = (rng.standard_normal((9, 11)) * np.exp(2 * rng.standard_normal((9, 1)))).astype(np.float32)
    x[0:2, 0:3] = 0.0  # an all-zero block -> scale_inv 1
    q, si = oracle.quantize_block(x, br, bc, fmt)
    wq, wsi = brute_force_block(x, br, bc, fmt)
    assert np.array_equal(si, wsi)
    assert np.array_equal(q, wq)
    if (br, bc) == (2, 3):
        assert si[0, 0] == 1.0


@pytest.mark.parametrize("br,bc", [(128, 128), (1, 128)])
def test_block_quantize_invariants(oracle, br, bc):
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((260, 300)) * 3).astype(np.float32)  # ragged edge blocks
    q, si = oracle.quantize_block(x, br, bc, E4M3)
    assert si.shape == (-(-260 // br), -(-300 // bc))
    # the element attaining each block's amax encodes to +-448
    for (i, j) in [(0, 0), (si.shape[0] - 1, si.shape[1] - 1), (si.shape[0] // 2, 1)]:
        blk = x[i * br:(i + 1) * br, j * bc:(j + 1) * bc]
        r, c = np.unravel_index(np.abs(blk).argmax(), blk.shape)
        assert q[i * br + r, j * bc + c] in (0x7E, 0xFE)
    # scaling by 2^k leaves codes unchanged and multiplies scale_inv by 2^k
    for k in (-7, 5):
        q2, si2 = oracle.quantize_block(x * np.float32(2.0 ** k), br, bc, E4M3)
        assert np.array_equal(q2, q)
        assert np.array_equal(si2, si * np.float32(2.0 ** k))
    q3, si3 = oracle.quantize_block(x, br, bc, E4M3, threads=3)
    assert np.array_equal(q3, q) and np.array_equal(si3, si)


# --------------------------------------------------------------- dequantize

@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_dequantize_matches_torch(oracle, fmt):
    rng = np.random.default_rng(4)
    q = rng.integers(0, 256, size=(64, 48), dtype=np.uint8)
    si = np.float32(0.0123)
    y = oracle.dequantize(q, fmt, np.array([si]), out_dt=oracle.BF16)
    prod = torch.from_numpy(q).view(TORCH_FP8[fmt]).float() * torch.tensor(si)
    want = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = torch.isnan(prod).numpy()
    assert np.array_equal(y[~nan], want[~nan])
    assert np.all(y[nan] == 0x7FFF)
    yf = oracle.dequantize(q, fmt, np.array([si]), out_dt=oracle.FP32)
    assert np.array_equal(yf[~nan], prod.numpy()[~nan])
    assert np.all(yf[nan].view(np.uint32) == 0x7FFFFFFF)


def test_block_dequantize_uses_each_blocks_scale(oracle):
    q = np.full((260, 300), 0x38, dtype=np.uint8)  # E4M3 0x38 = 1.0
    for br, bc in [(128, 128), (1, 128)]:
        nbr, nbc = -(-260 // br), -(-300 // bc)
        si = (2.0 ** np.arange(nbr * nbc).reshape(nbr, nbc) % 29).astype(np.float32) + 1
        y = oracle.dequantize(q, E4M3, si, br, bc, out_dt=oracle.FP32)
        want = np.repeat(np.repeat(si, br, 0), bc, 1)[:260, :300]
        assert np.array_equal(y, want)
        y3 = oracle.dequantize(q, E4M3, si, br, bc, out_dt=oracle.FP32, threads=3)
        assert np.array_equal(y3, y)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_quantize_dequantize_round_trip(oracle, fmt):
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.decode(codes, fmt)
    keep = ~np.isnan(dec)
    for si in (1.0, 0.0078125, 3.3, 1e-3):
        s = np.float32(1.0) / np.float32(si)
        y = oracle.dequantize(codes[keep], fmt, np.array([si], np.float32), out_dt=oracle.FP32)
        back, _ = oracle.quantize(y.ravel(), fmt, s)
        assert np.array_equal(back, codes[keep])


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_sqnr_soft_check(oracle, fmt):
    g = golden("error_bounds.txt")
    rule = g["e4m3.sqnr_rule_db" if fmt == E4M3 else "e5m2.sqnr_rule_db"]
    assert abs(rule - (6.02 * MANT[fmt] + 1.76)) < 0.01
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200_000).astype(np.float32)
    s, si = oracle.compute_scale(oracle.amax(x), fmt, 0)
    q, _ = oracle.quantize(x, fmt, s)
    y = oracle.dequantize(q, fmt, np.array([si]), out_dt=oracle.FP32).ravel().astype(np.float64)
    sqnr = 10 * np.log10(np.mean(x.astype(np.float64) ** 2) / np.mean((x - y) ** 2))
    assert sqnr > rule  # floating-point grids do at least as well as the uniform rule of thumb


# ------------------------------------------------------------------ hybrid

def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_hybrid_same_format_original_is_cast_transpose(oracle):
    rng = np.random.default_rng(21)
    bits = _bf16(rng.standard_normal((37, 45)) * 20)
    for fmt in (E4M3, E5M2):
        s = np.float32(3.5)
        qr, qc = oracle.quantize_hybrid(bits, fmt, s, fmt, s, oracle.SRC_ORIGINAL)
        wr, wc = oracle.cast_transpose(bits, fmt, s)
        assert np.array_equal(qr, wr) and np.array_equal(qc, wc)


def test_hybrid_cross_format_directions_are_independent(oracle):
    rng = np.random.default_rng(22)
    bits = _bf16(rng.standard_normal((40, 24)) * 300)
    sr, sc = np.float32(1.25), np.float32(0.03)
    qr, qc = oracle.quantize_hybrid(bits, E4M3, sr, E5M2, sc, oracle.SRC_ORIGINAL)
    assert np.array_equal(qr, oracle.quantize(bits, E4M3, sr)[0])
    assert np.array_equal(qc, oracle.quantize(np.ascontiguousarray(bits.T), E5M2, sc)[0])


def test_hybrid_rowwise_dequantized_source(oracle):
    rng = np.random.default_rng(23)
    bits = _bf16(rng.standard_normal((33, 50)) * 7)
    sr = np.float32(17.0)
    # same format and scale: re-quantizing the dequantized value gives the rowwise codes back
    qr, qc = oracle.quantize_hybrid(bits, E4M3, sr, E4M3, sr, oracle.SRC_ROWWISE_DEQUANTIZED)
    assert np.array_equal(qc, qr.T)
    # the columnwise source is exactly the BF16 dequantized rowwise tensor (the documented reading)
    sc = np.float32(0.5)
    qr, qc = oracle.quantize_hybrid(bits, E4M3, sr, E5M2, sc, oracle.SRC_ROWWISE_DEQUANTIZED)
    y = oracle.dequantize(qr, E4M3, np.array([np.float32(1.0) / sr]), out_dt=oracle.BF16)
    assert np.array_equal(qc, oracle.quantize(np.ascontiguousarray(y.T), E5M2, sc)[0])
    # E4M3 -> E5M2 from the coarser rowwise grid differs from quantizing the original
    _, qc_orig = oracle.quantize_hybrid(bits, E4M3, sr, E5M2, sc, oracle.SRC_ORIGINAL)
    assert not np.array_equal(qc, qc_orig)
