"""Host-side logic that needs no GPU: the C ABI library loads and exports every
entry point its header declares, argument validation rejects bad calls
before touching a device, the byte accounting of the benchmark, the
multi-rank reduction over gloo, and the reference arm's JSON line."""
from __future__ import annotations

import ctypes
import json
import os
import subprocess
import sys

import pytest
import torch

import fp8_scaled_quantization_gb300 as fq
from fp8_scaled_quantization_gb300 import _lib
from conftest import ROOT


def test_library_exports_every_header_symbol(native_lib):
    names = _lib.header_entry_points()
    assert {"fp8_amax", "fp8_update_scale_delayed", "fp8_quantize", "fp8_quantize_cast_transpose",
            "fp8_quantize_block", "fp8_dequantize"} <= set(names)
    raw = ctypes.CDLL(_lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(names) <= set(_lib.SIGNATURES), "every declared entry point has a binding signature"


def test_library_built_for_sm103a(native_lib):
    from fp8_scaled_quantization_gb300 import build as b
    assert "arch=compute_103a,code=sm_103a" in b.ARCH
    assert "-ffast-math" not in b.NVCC_FLAGS and "--use_fast_math" not in b.NVCC_FLAGS


def test_status_strings_and_version(native_lib):
    assert native_lib.fp8_status_string(0) == b"FP8_OK"
    assert native_lib.fp8_status_string(2) == b"FP8_ERR_UNSUPPORTED"
    assert native_lib.fp8_version() == (0 << 16) | 1


BAD = 0x1000  # never dereferenced: every call below is rejected on the host first


@pytest.mark.parametrize("call,status,msg", [
    (lambda L: L.fp8_quantize(BAD, 0, 10, 9, BAD, BAD, None, None, None), 1, "unknown format"),
    (lambda L: L.fp8_quantize(BAD, 5, 10, 0, BAD, BAD, None, None, None), 1, "unknown dtype"),
    (lambda L: L.fp8_quantize(BAD, 0, -1, 0, BAD, BAD, None, None, None), 1, "n < 0"),
    (lambda L: L.fp8_quantize(BAD, 0, 10, 0, None, BAD, None, None, None), 1, "scale is NULL"),
    (lambda L: L.fp8_quantize(BAD + 1, 0, 10, 0, BAD, BAD, None, None, None), 1, "element-aligned"),
    (lambda L: L.fp8_amax(BAD, 0, 10, None, 0, 0, None, None, None), 1, "amax_out is NULL"),
    (lambda L: L.fp8_amax(BAD, 0, 10, BAD, 0, 0, BAD, None, None), 1, "both"),
    (lambda L: L.fp8_amax(BAD, 0, 10, BAD, 0, 127, BAD, BAD, None), 1, "margin"),
    (lambda L: L.fp8_update_scale_delayed(BAD, 0, 0, None, 0, 0, 0, BAD, BAD, None), 1, "history_len"),
    (lambda L: L.fp8_update_scale_delayed(BAD, 4, -1, None, 0, 0, 0, BAD, BAD, None), 1, "step < 0"),
    (lambda L: L.fp8_update_scale_delayed(BAD, 4, 0, None, 3, 0, 0, BAD, BAD, None), 1, "unknown algo"),
    (lambda L: L.fp8_update_scale_delayed(BAD, 4, 0, None, 0, 0, 0, None, BAD, None), 1, "NULL"),
    (lambda L: L.fp8_quantize_delayed(BAD, 0, 10, 0, BAD, BAD, BAD, BAD, 0, 0, 0, 0, None, None, None), 1,
     "history_len"),
    (lambda L: L.fp8_quantize_delayed(BAD, 0, 10, 0, None, BAD, BAD, BAD, 4, 0, 0, 0, None, None, None), 1,
     "scale / scale_inv is NULL"),
    (lambda L: L.fp8_quantize_delayed(BAD, 0, 10, 0, BAD, BAD, BAD, BAD, 4, 0, 2, 0, None, None, None), 1,
     "unknown algo"),
    (lambda L: L.fp8_quantize_cast_transpose(BAD, 0, 4, 4, 0, BAD, None, None, None, None), 1, "both NULL"),
    (lambda L: L.fp8_quantize_cast_transpose(BAD, 0, -4, 4, 0, BAD, BAD, None, None, None), 1, "negative"),
    (lambda L: L.fp8_quantize_block(BAD, 0, 4, 4, 64, 64, 0, BAD, BAD, None), 2, "block shape"),
    (lambda L: L.fp8_quantize_block(BAD, 0, 4, 4, 128, 1, 0, BAD, BAD, None), 2, "block shape"),
    (lambda L: L.fp8_quantize_block(BAD, 0, 4, 4, 128, 128, 0, None, BAD, None), 1, "NULL"),
    (lambda L: L.fp8_dequantize(BAD, 0, 4, 4, BAD, 32, 32, BAD, 0, None), 2, "block shape"),
    (lambda L: L.fp8_dequantize(BAD, 0, 4, 4, BAD, 0, 0, BAD, 7, None), 1, "out_dtype"),
    (lambda L: L.fp8_dequantize(BAD, 0, 4, 4, BAD + 2, 0, 0, BAD, 0, None), 1, "scale_inv not 4-byte"),
    (lambda L: L.fp8_quantize_current(BAD, 0, -1, 0, 0, BAD, None, None, None, None), 1, "n < 0"),
    (lambda L: L.fp8_quantize_current(BAD, 0, 10, 0, 200, BAD, None, None, None, None), 1, "margin"),
    (lambda L: L.fp8_quantize_current(BAD, 0, 10, 4, 0, BAD, None, None, None, None), 1, "unknown format"),
    (lambda L: L.fp8_quantize_current(None, 0, 10, 0, 0, BAD, None, None, None, None), 1, "is NULL"),
    (lambda L: L.fp8_quantize_hybrid(BAD, 0, 4, 4, 0, BAD, BAD, 1, BAD, BAD, 5, None), 1, "columnwise source"),
    (lambda L: L.fp8_quantize_hybrid(BAD, 0, 4, 4, 0, BAD, BAD, 3, BAD, BAD, 0, None), 1, "unknown format"),
    (lambda L: L.fp8_quantize_hybrid(BAD, 0, 4, 4, 0, None, BAD, 1, BAD, BAD, 0, None), 1, "scale is NULL"),
    (lambda L: L.fp8_quantize_hybrid(BAD, 0, 4, 4, 0, BAD, None, 1, BAD, BAD, 1, None), 1, "q_col is NULL"),
    (lambda L: L.fp8_quantize_block_cast_transpose(BAD, 0, 4, 4, 0, BAD, None, None, None, None), 1,
     "both its codes and its scales"),
    (lambda L: L.fp8_quantize_block_cast_transpose(BAD, 0, 4, 4, 0, None, None, None, None, None), 1,
     "no output requested"),
    (lambda L: L.fp8_quantize_block_cast_transpose(BAD, 0, 4, 4, 0, BAD, BAD + 2, None, None, None), 1,
     "not 4-byte aligned"),
    (lambda L: L.fp8_amax_grouped(0, BAD, BAD, 0, BAD, 0, 0, None, None, None), 1, "count must be"),
    (lambda L: L.fp8_amax_grouped(129, BAD, BAD, 0, BAD, 0, 0, None, None, None), 1, "count must be"),
    (lambda L: L.fp8_amax_grouped(2, BAD, BAD, 0, None, 0, 0, None, None, None), 1, "no output requested"),
    (lambda L: L.fp8_quantize_grouped(2, None, BAD, 0, 0, BAD, BAD, None), 1, "is NULL"),
    (lambda L: L.fp8_quantize_grouped(2, BAD, BAD, 0, 0, None, BAD, None), 1, "scales is NULL"),
    (lambda L: L.fp8_wait_timeouts(None), 1, "count is NULL"),
])
def test_host_validation_rejects_before_launch(native_lib, call, status, msg):
    before = native_lib.fp8_launch_count()
    assert call(native_lib) == status
    assert msg in native_lib.fp8_last_error_message().decode()
    assert native_lib.fp8_launch_count() == before


def test_empty_inputs_need_no_device(native_lib):
    # nothing to do and no reduction requested: success without touching CUDA
    assert native_lib.fp8_quantize(None, 0, 0, 0, BAD, None, None, None, None) == 0
    assert native_lib.fp8_quantize_block(None, 0, 0, 128, 128, 128, 0, None, None, None) == 0
    assert native_lib.fp8_dequantize(None, 0, 0, 5, None, 0, 0, None, 0, None) == 0


def test_binding_rejects_host_and_strided_tensors(native_lib):
    x = torch.zeros(16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fq.fp8_quantize(x, fq.E4M3, torch.ones(1), torch.empty(16, dtype=torch.uint8))
    with pytest.raises(TypeError):
        fq.fp8_quantize(x, fq.E4M3, torch.ones(1), torch.empty(16, dtype=torch.int8))


def test_library_missing_fails_loudly(tmp_path):
    with pytest.raises(_lib.LibraryMissing):
        saved = _lib._lib
        try:
            _lib._lib = None
            _lib.load(str(tmp_path / "nope.so"))
        finally:
            _lib._lib = saved


# ------------------------------------------------------------ byte accounting

def test_pipeline_byte_accounting_full_size():
    import bench
    from fp8_scaled_quantization_gb300 import pipelines as P
    shapes = bench.workload_shapes(1.0)
    meta = torch.device("meta")
    mk = lambda s: torch.empty(s, dtype=torch.bfloat16, device=meta)  # noqa: E731
    inp = {"w1": mk(shapes["w1"]), "w2": mk(shapes["w2"]), "w3": [mk(shapes["w3"]) for _ in range(16)],
           "w4": (mk(shapes["w4w"]), mk(shapes["w4a"])), "w5": [mk(shapes["w5"]) for _ in range(32)]}
    pipes = bench.make_pipelines(inp)
    b = {k: p.bytes() for k, p in pipes.items()}
    N1, N2, N3, N5 = 1024 * 1024, 8192 * 8192, 4096 * 14336, 8192 * 8192
    assert b["W1"].total == 5 * N1
    assert b["W2"].total == 6 * N2
    assert b["W3"].per_kernel["quantize_delayed"] == (16 * (3 * N3 + 4 * 1024 + 12), 16)
    assert b["W4"].per_kernel["block128x128"][0] == 3 * 7168 * 18432 + 4 * 56 * 144
    assert b["W4"].per_kernel["block1x128"][0] == 3 * 16384 * 7168 + 4 * 16384 * 56
    assert b["W5"].total == 32 * 8 * N5
    total = sum(x.total for x in b.values())
    assert 21.0e9 < total < 21.3e9
    w5 = b["W5"].per_kernel
    if bench.W5_GROUP == "all":
        assert w5["amax_grouped"] == (32 * 2 * N5, 1) and w5["quantize_grouped"] == (32 * 3 * N5, 1)
        w5_calls = 1 + 1 + 32
    elif bench.W5_GROUP == "amax":
        assert w5["amax_grouped"] == (32 * 2 * N5, 1) and w5["quantize"] == (32 * 3 * N5, 32)
        w5_calls = 1 + 32 + 32
    else:
        assert w5["quantize_current"] == (32 * 5 * N5, 32)
        w5_calls = 32 + 32
    assert w5["dequantize"] == (32 * 3 * N5, 32)
    assert sum(x.launches for x in b.values()) == 1 + 2 + (16 + 1) + 2 + w5_calls  # API calls


# ------------------------------------------------------------- multi-rank

def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(10.0 + 5 * rank, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import socket
    import torch.multiprocessing as mp
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_reference_arm_line_shape():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--scale", "0.125"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_grouped_binding_marshals_and_rejects_host_tensors():
    """The grouped bindings build their host pointer / size tables before the
    device check rejects CPU tensors (no CUDA call is made)."""
    import fp8_scaled_quantization_gb300 as fq
    xs = [torch.zeros(16, dtype=torch.bfloat16), torch.zeros(32, dtype=torch.bfloat16)]
    with pytest.raises(ValueError, match="CUDA device"):
        fq.fp8_amax_grouped(xs, torch.zeros(2))
    with pytest.raises(ValueError, match="CUDA device"):
        fq.fp8_quantize_grouped(xs, fq.E4M3, torch.zeros(2), [torch.zeros(16, dtype=torch.uint8),
                                                               torch.zeros(32, dtype=torch.uint8)])
    with pytest.raises(ValueError, match="at least len"):
        fq.fp8_amax_grouped(xs, torch.zeros(1))


def test_two_call_current_scaling_byte_accounting():
    from fp8_scaled_quantization_gb300 import pipelines as P
    x = torch.empty((1024, 1024), dtype=torch.bfloat16, device=torch.device("meta"))
    b = P.CurrentScaling(x, current_call=False).bytes()
    assert b.per_kernel == {"amax": (2 * 2 ** 20, 1), "quantize": (3 * 2 ** 20, 1)}
    g = P.GradientQDQ([x, x], current_call=False).bytes()
    assert g.per_kernel["amax"] == (2 * 2 * 2 ** 20, 2) and g.per_kernel["dequantize"] == (2 * 3 * 2 ** 20, 2)
    c = P.GradientQDQ([x, x]).bytes()
    assert c.per_kernel["quantize_current"] == (2 * 5 * 2 ** 20, 2)


def test_input_digests_hash_each_workloads_bytes():
    import hashlib
    import bench
    g = torch.Generator().manual_seed(0)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    inp = {"w1": mk(4, 8), "w2": mk(8, 8), "w3": [mk(2, 8), mk(2, 8)], "w4": (mk(4, 4), mk(2, 4)), "w5": [mk(3, 8)]}
    d = bench.input_digests(inp)
    h = hashlib.sha256()
    for t in inp["w3"]:
        h.update(t.view(torch.int16).numpy().tobytes())
    assert d["W3"] == h.hexdigest()[:16]
    assert set(d) == {"W1", "W2", "W3", "W4", "W5"} and len(set(d.values())) == 5


def test_bench_parity_check_reports_bit_exact_and_mismatches():
    """bench.py checks the timed step's outputs against the oracle's in its CPU
    baseline leg: identical outputs read bit-exact, one flipped byte is named."""
    import copy
    import numpy as np
    import bench
    from fp8_scaled_quantization_gb300 import workloads as wl
    inp = {"w1": wl.w1_outliers((64, 128)), "w2": wl.w2_student_t((128, 256)),
           "w3": list(wl.w3_steps((64, 256), 3)), "w4": wl.w4_block((256, 256), (64, 384)),
           "w5": list(wl.w5_gradients((64, 512), 2))}
    host = bench.host_sample(inp, 1.0, max_w3=3, max_w5=2)
    ref = {}
    nbytes = bench.oracle_suite_sample(host, 1.0, 2, ref)
    assert nbytes > 0 and set(ref) == {"W1", "W2", "W3", "W4", "W5"}
    snap = {w: {k: np.array(v, copy=True).reshape(-1) if np.ndim(v) == 0 else np.array(v, copy=True)
                for k, v in d.items()} for w, d in ref.items()}
    out = bench.compare_parity(snap, ref)
    assert all(out[w] == "bit-exact" for w in ("W1", "W2", "W3", "W4", "W5")), out
    bad = copy.deepcopy(snap)
    bad["W4"]["q_a"].reshape(-1)[17] ^= 1
    bad["W3"]["sat"][1] += 1
    out = bench.compare_parity(bad, ref)
    assert out["W4"] == "MISMATCH: q_a" and out["W3"] == "MISMATCH: sat" and out["W1"] == "bit-exact"
