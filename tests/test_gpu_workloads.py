"""Full-size parity: the five benchmark workloads, run through the same
pipelines (and so the same launch configurations) that bench.py times, each
checked against the CPU oracle on the same bytes.  The oracle runs its plain
C loops on disjoint row ranges in threads."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_scaled_quantization_gb300 as fq
from fp8_scaled_quantization_gb300 import pipelines as P
from fp8_scaled_quantization_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def bench_w5_group():
    import bench
    return bench.W5_GROUP


def bits(x):
    return wl.bf16_bits(x)


def f32b(t):
    return t.detach().cpu().numpy().view(np.uint32)


@pytest.fixture(scope="module")
def threads(oracle):
    return oracle.default_threads()


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_w1_current_e4m3_1024(cuda, oracle, threads):
    x = wl.w1_outliers(device=cuda)
    p = P.CurrentScaling(x, fq.E4M3, 0)
    p.run()
    torch.cuda.synchronize()
    xb = bits(x)
    amax = oracle.amax(xb, threads)
    assert amax == np.float32(2000.0)  # the planted outliers set the amax exactly
    s, si = oracle.compute_scale(amax, oracle.E4M3, 0)
    assert f32b(p.amax)[0] == np.float32(amax).view(np.uint32)
    assert (f32b(p.scale)[0], f32b(p.scale_inv)[0]) == (s.view(np.uint32), si.view(np.uint32))
    q, _ = oracle.quantize(xb, oracle.E4M3, s, threads)
    assert np.array_equal(p.q.cpu().numpy(), q)


def test_w2_cast_transpose_8192(cuda, oracle, threads):
    x = wl.w2_student_t(device=cuda)
    p = P.CurrentCastTranspose(x, fq.E4M3, 1)
    p.run()
    torch.cuda.synchronize()
    xb = bits(x)
    s, si = oracle.compute_scale(oracle.amax(xb, threads), oracle.E4M3, 1)
    assert (f32b(p.scale)[0], f32b(p.scale_inv)[0]) == (s.view(np.uint32), si.view(np.uint32))
    qr, qc = oracle.cast_transpose(xb, oracle.E4M3, s, threads)
    assert np.array_equal(p.q_row.cpu().numpy(), qr)
    assert np.array_equal(p.q_col.cpu().numpy(), qc)


def test_w3_delayed_16_steps(cuda, oracle, threads):
    xs = list(wl.w3_steps(device=cuda))
    p = P.DelayedScaling(xs, 1024, fq.E4M3, 0, keep_codes=True, record_scales=True)
    p.run()
    torch.cuda.synchronize()
    hist = np.zeros(1024, np.float32)
    s, si = oracle.update_delayed(hist, 0, None, oracle.ALGO_MAX, oracle.E4M3, 0)
    scales, amaxes, sats = f32b(p.scales), f32b(p.amax), p.sat.cpu().numpy()
    total_sat = 0
    for k, x in enumerate(xs):
        xb = bits(x)
        assert scales[k] == s.view(np.uint32), k
        q, sat = oracle.quantize(xb, oracle.E4M3, s, threads)
        assert np.array_equal(p.q[k].cpu().numpy(), q), k
        assert sats[k] == sat, k
        a = oracle.amax(xb, threads)
        assert amaxes[k] == np.float32(a).view(np.uint32)
        s, si = oracle.update_delayed(hist, k, a, oracle.ALGO_MAX, oracle.E4M3, 0)
        total_sat += sat
    assert (f32b(p.scale)[0], f32b(p.scale_inv)[0]) == (s.view(np.uint32), si.view(np.uint32))
    assert np.array_equal(f32b(p.hist), hist.view(np.uint32))
    assert total_sat > 0  # the growing magnitudes overflow the one-step-stale scale


def test_w4_blockwise(cuda, oracle, threads):
    w, a = wl.w4_block(device=cuda)
    p = P.BlockScaling(w, a, fq.E4M3)
    p.run()
    torch.cuda.synchronize()
    qw, siw = oracle.quantize_block(bits(w), 128, 128, oracle.E4M3, threads)
    assert np.array_equal(f32b(p.si_w), siw.view(np.uint32))
    assert np.array_equal(p.q_w.cpu().numpy(), qw)
    del qw
    qa, sia = oracle.quantize_block(bits(a), 1, 128, oracle.E4M3, threads)
    assert np.array_equal(f32b(p.si_a), sia.view(np.uint32))
    assert np.array_equal(p.q_a.cpu().numpy(), qa)


def test_w5_e5m2_quantize_dequantize(cuda, oracle, threads):
    """Every element of all 32 gradient tensors: scale, codes and dequantized BF16."""
    xs = list(wl.w5_gradients(device=cuda))
    p = P.GradientQDQ(xs, fq.E5M2, 0, keep_outputs=True, group=bench_w5_group())  # as the bench runs it
    p.run()
    torch.cuda.synchronize()
    scales, scale_invs, amaxes = f32b(p.scale), f32b(p.scale_inv), f32b(p.amax)
    for k, x in enumerate(xs):
        xb = bits(x)
        a = oracle.amax(xb, threads)
        s, si = oracle.compute_scale(a, oracle.E5M2, 0)
        assert amaxes[k] == np.float32(a).view(np.uint32), k
        assert (scales[k], scale_invs[k]) == (s.view(np.uint32), si.view(np.uint32)), k
        q, _ = oracle.quantize(xb, oracle.E5M2, s, threads)
        assert np.array_equal(p.q[k].cpu().numpy(), q), k
        y = oracle.dequantize(q, oracle.E5M2, np.array([si]), threads=threads)
        assert np.array_equal(bits(p.y[k]), y), k
        del xb, q, y


@pytest.mark.parametrize("group", ["", "amax", "all"])
def test_w5_pipeline_orders_agree(cuda, oracle, group):
    """The three ways GradientQDQ can organise the per-tensor current scaling
    give the same scales, codes and dequantized values (small tensors)."""
    g = torch.Generator(device="cpu").manual_seed(77)
    xs = [(torch.randn((257, 384), generator=g) * (10.0 ** k)).to(torch.bfloat16).to(cuda) for k in range(-2, 3)]
    p = P.GradientQDQ(xs, fq.E5M2, 1, keep_outputs=True, group=group)
    p.run()
    torch.cuda.synchronize()
    for k, x in enumerate(xs):
        xb = bits(x)
        s, si = oracle.compute_scale(oracle.amax(xb), oracle.E5M2, 1)
        assert f32b(p.scale)[k] == s.view(np.uint32) and f32b(p.scale_inv)[k] == si.view(np.uint32), k
        q, _ = oracle.quantize(xb, oracle.E5M2, s)
        assert np.array_equal(p.q[k].cpu().numpy(), q), k
        assert np.array_equal(bits(p.y[k]), oracle.dequantize(q, oracle.E5M2, np.array([si]))), k
