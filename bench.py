"""Throughput benchmark of the GB300 FP8 scaled-quantization library.

One step = one pass of the whole hot path over the five synthetic workloads
(each kernel of the library runs in it):
  W1 current scaling E4M3, BF16 1024x1024               amax(+scale) -> quantize
  W2 current scaling cast+transpose E4M3, 8192x8192     amax(+scale) -> cast_transpose
  W3 delayed scaling E4M3, 16 steps of 4096x14336       quantize (+ amax, sat, history update) x16
  W4 blockwise E4M3, 128x128 on 7168x18432, 1x128 on 16384x7168
  W5 E5M2 current scaling + dequantize, 32 x 8192x8192  grouped amax(+scale, per-tensor scales)
                                                       -> (quantize -> dequantize) x32
value = compulsory bytes (each workload's inputs read once and outputs written
once; the amax passes of current scaling are not counted) / time, in GB/s,
with inputs resident in HBM.  The inputs (~6.5 GB) and the step's traffic
(~21 GB) are far larger than the 135 MB L2, so no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workloads (the method has no other implementation
to compare with).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantize GB/s (bytes read+written) and % of GB300 HBM peak per cast variant"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_NAME = ("fp8 scaled-quantization suite: W1 current E4M3 1024x1024; W2 current cast+transpose E4M3 "
                 "8192x8192 margin 1; W3 delayed E4M3 16 x 4096x14336 hist 1024; W4 block E4M3 128x128 "
                 "7168x18432 + 1x128 16384x7168; W5 current E5M2 quantize+dequantize 32 x 8192x8192")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="shrink every workload's row count by this factor (testing only; 1.0 = full size)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the separately timed kernels beyond the step")
    ap.add_argument("--extras-only", action="store_true",
                    help="time only the separately timed kernels (MXFP8, hybrid, block cast-transpose, grouped)")
    ap.add_argument("--cpu-fraction", type=float, default=1.0,
                    help="fraction of each workload's rows the CPU-oracle baseline processes")
    ap.add_argument("--workloads", default="W1,W2,W3,W4,W5",
                    help="comma-separated subset of W1..W5 (profiling a single workload)")
    ap.add_argument("--count", type=int, default=0,
                    help="cap on W3 steps and W5 tensors (0 = the full 16 / 32; profiling only)")
    ap.add_argument("--nvtx", action="store_true",
                    help="an NVTX range around every workload of every step (for a timeline profiler)")
    return ap.parse_args()


# ----------------------------------------------------------------- workloads

def workload_shapes(scale: float, count: int = 0):
    from fp8_scaled_quantization_gb300 import workloads as wl

    def s(shape, mult=128):
        r = max(mult, int(shape[0] * scale) // mult * mult)
        return (r, shape[1])

    return {
        "w1": wl.W1_SHAPE,
        "w2": s(wl.W2_SHAPE),
        "w3": s(wl.W3_SHAPE),
        "w4w": s(wl.W4_WEIGHT_SHAPE),
        "w4a": s(wl.W4_ACT_SHAPE),
        "w5": s(wl.W5_SHAPE),
        "w3_steps": min(wl.W3_STEPS, count) if count > 0 else wl.W3_STEPS,
        "w5_count": min(wl.W5_TENSORS, count) if count > 0 else wl.W5_TENSORS,
    }


ALL_WORKLOADS = ("W1", "W2", "W3", "W4", "W5")


def make_inputs(shapes, device, seed_offset=0, which=ALL_WORKLOADS):
    from fp8_scaled_quantization_gb300 import workloads as wl
    S = wl.SEEDS
    inp = {}
    if "W1" in which:
        inp["w1"] = wl.w1_outliers(shapes["w1"], device, seed=S["w1"] + seed_offset)
    if "W2" in which:
        inp["w2"] = wl.w2_student_t(shapes["w2"], device, seed=S["w2"] + seed_offset)
    if "W3" in which:
        inp["w3"] = list(wl.w3_steps(shapes["w3"], shapes["w3_steps"], device, seed=S["w3"] + seed_offset))
    if "W4" in which:
        inp["w4"] = wl.w4_block(shapes["w4w"], shapes["w4a"], device, seed=S["w4"] + seed_offset)
    if "W5" in which:
        inp["w5"] = list(wl.w5_gradients(shapes["w5"], shapes["w5_count"], device, seed=S["w5"] + seed_offset))
    return inp


def make_pipelines(inp):
    from fp8_scaled_quantization_gb300 import pipelines as P, E4M3, E5M2
    pipes = {}
    if "w1" in inp:
        pipes["W1"] = P.CurrentScaling(inp["w1"], E4M3, 0)
    if "w2" in inp:
        pipes["W2"] = P.CurrentCastTranspose(inp["w2"], E4M3, 1)
    # Every W3 step and every W5 tensor writes its own output buffers: with one
    # buffer reused, a launch would overwrite lines of the previous launch's
    # output that are still dirty in L2, and those writes would never reach
    # DRAM (the delayed cast measured 27.5 against 31.4 us back to back).
    if "w3" in inp:
        pipes["W3"] = P.DelayedScaling(inp["w3"], 1024, E4M3, 0, keep_codes=True)
    if "w4" in inp:
        pipes["W4"] = P.BlockScaling(*inp["w4"], E4M3)
    if "w5" in inp:
        pipes["W5"] = P.GradientQDQ(inp["w5"], E5M2, 0, keep_outputs=True, group=W5_GROUP)
    return pipes


# --------------------------------------------------------------------- timing

class EventTimer:
    """CUDA events around each launch, per kernel name (current stream)."""

    def __init__(self):
        import torch
        self.torch = torch
        self.pool = []
        self.spans = {}
        self.open = {}

    def _ev(self):
        return self.pool.pop() if self.pool else self.torch.cuda.Event(enable_timing=True)

    def reserve(self, n):
        self.pool.extend(self.torch.cuda.Event(enable_timing=True) for _ in range(n))

    def start(self, name):
        e = self._ev()
        e.record()
        self.open[name] = e

    def stop(self, name):
        e = self._ev()
        e.record()
        self.spans.setdefault(name, []).append((self.open.pop(name), e))

    def totals(self):
        """name -> (total ms, launches); call after a synchronize."""
        return {k: (sum(a.elapsed_time(b) for a, b in v), len(v)) for k, v in self.spans.items()}

    def medians(self):
        """name -> median ms of one bracketed call; call after a synchronize."""
        return {k: statistics.median(a.elapsed_time(b) for a, b in v) for k, v in self.spans.items()}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.proc, self.path, self.gpu_id = None, None, gpu_id

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() in ("active", "1", "yes")})
        load = [v for v in sm if v and mx and v > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# How the W5 tensors' current scaling is organised (GradientQDQ's `group`):
# one grouped amax + scale call for the 32 tensors, then per tensor the cast
# and its dequantize (which reads the codes while they are still in L2).
# Measured on the step: 5303 GB/s, against 5174 with fp8_quantize_current per
# tensor and 5187 with the cast grouped as well.
W5_GROUP = "amax"

SINGLE_KERNEL_CALLS = ("quantize", "quantize_grouped", "cast_transpose", "block128x128", "block1x128", "dequantize")


def kernel_traffic(kernel: str):
    """DRAM bytes per element from the committed ncu summary, when it was taken
    on the current source of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    src = {"quantize": "quantize.cu", "quantize_delayed": "quantize.cu", "cast_transpose": "cast_transpose.cu",
           "quantize_grouped": "grouped.cu",
           "amax": "amax_scale.cu",
           "dequantize": "dequantize.cu", "block128x128": "block_quant.cu", "block1x128": "block_quant.cu"}.get(kernel)
    if src is None or not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in (src, "fp8q_device.cuh"):
        h.update(open(os.path.join(ROOT, "fp8_scaled_quantization_gb300", "csrc", f), "rb").read())
    digest = h.hexdigest()[:16]
    for line in open(path):
        m = dict(re.findall(r"(\w+)=(\S+)", line))
        if m.get("kernel") == kernel and m.get("source_sha") == digest:
            return float(m["dram_bytes_per_element"])
    return None


# ------------------------------------------------------------------ our arm

def compulsory_bytes(pipes) -> int:
    """Bytes each workload must move at least: its inputs read once and its
    outputs written once (amax passes and re-reads not counted)."""
    total = 0
    for name, p in pipes.items():
        if name == "W1":
            total += p.x.numel() * (p.x.element_size() + 1)
        elif name == "W2":
            total += p.x.numel() * (p.x.element_size() + 2)
        elif name == "W3":
            total += sum(x.numel() * (x.element_size() + 1) for x in p.xs)
        elif name == "W4":
            total += p.bytes().total
        elif name == "W5":
            total += sum(x.numel() * (x.element_size() + 1 + 1 + 2) for x in p.xs)
    return total


def run_ours(args, rank, world):
    import torch
    import fp8_scaled_quantization_gb300 as fq
    from fp8_scaled_quantization_gb300.pipelines import KernelBytes

    fq.library()  # raises if the CUDA library is missing: there is no fallback
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    shapes = workload_shapes(args.scale, args.count)
    which = tuple(w.strip().upper() for w in args.workloads.split(",") if w.strip())
    full_suite = set(which) == set(ALL_WORKLOADS) and args.scale == 1.0 and args.count == 0
    inp = make_inputs(shapes, dev, seed_offset=rank, which=which)
    pipes = make_pipelines(inp)
    per_variant_bytes = {k: p.bytes() for k, p in pipes.items()}
    kb = KernelBytes()
    for b in per_variant_bytes.values():
        for name, (nbytes, launches) in b.per_kernel.items():
            kb.add(name, nbytes // launches, launches)
    kernel_bytes = kb.total
    step_bytes = compulsory_bytes(pipes)
    torch.cuda.synchronize()

    def step(timer=None, vt=None):
        for name, p in pipes.items():
            if args.nvtx:
                torch.cuda.nvtx.range_push(name)
            if vt is not None:
                vt.start(name)
            p.run(timer)
            if vt is not None:
                vt.stop(name)
            if args.nvtx:
                torch.cuda.nvtx.range_pop()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_uuid = gpu_uuid if gpu_uuid.startswith("GPU-") else "GPU-" + gpu_uuid
    except Exception:
        pass
    clocks = ClockSampler(gpu_uuid)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    launches0 = fq.launch_count()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        step()
    t1.record()
    torch.cuda.synchronize()
    launches = fq.launch_count() - launches0
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1)
    ms_max = max_over_ranks(ms, world)

    # The headline region carries only its two bracketing events.  An event
    # recorded between two launches ends programmatic dependent launch there:
    # the second kernel can no longer become resident while the first drains,
    # and its dispatch latency lands inside the measured interval.  So each
    # breakdown gets a pass of its own right after the timed region:
    #   variants  -- events only at workload boundaries;
    #   kernels   -- back to back: each call repeated between two events (its
    #                steady-state duration on the stream, launches still chained),
    #                and, as an upper bound, events around every launch of a step.
    ksteps = max(3, min(args.steps, 20))
    peak, peak_kind = measured_hbm_peak()
    vtimer = EventTimer()
    vtimer.reserve(2 * len(pipes) * ksteps + 8)
    for _ in range(ksteps):
        step(vt=vtimer)
    torch.cuda.synchronize()
    variants = {}
    for name, (tot_ms, n) in vtimer.totals().items():
        cb = compulsory_bytes({name: pipes[name]})
        gbs = cb * ksteps / (tot_ms * 1e-3) / 1e9
        kbv = per_variant_bytes[name].total
        variants[name] = {"compulsory_bytes": cb, "kernel_bytes": kbv,
                          "ms_per_step": round(tot_ms / ksteps, 4), "gbs": round(gbs, 1),
                          "frac": round(gbs / peak, 4),
                          "kernel_gbs": round(kbv * ksteps / (tot_ms * 1e-3) / 1e9, 1),
                          "kernel_frac": round(kbv * ksteps / (tot_ms * 1e-3) / 1e9 / peak, 4)}

    timer = EventTimer()
    timer.reserve(2 * kb.launches * ksteps + 8)
    for _ in range(ksteps):
        step(timer)
    torch.cuda.synchronize()
    medians = timer.medians()
    kernels = {}
    for name, (tot_ms, n) in timer.totals().items():
        nbytes, nl = kb.per_kernel[name]
        kernels[name] = {"launches_per_step": nl, "bytes_per_step": nbytes,
                         "bytes_per_launch": round(nbytes / nl),
                         "bracketed_avg_us": round(tot_ms * 1e3 / n, 2),
                         "bracketed_median_us": round(medians[name] * 1e3, 2)}
    snap = snapshot_outputs(pipes) if full_suite else None

    for name, (fn, nbytes) in back_to_back_calls(pipes, dev).items():
        if name not in kernels:
            continue
        small = nbytes < B2B_GRAPH_BELOW_BYTES
        us = time_back_to_back(fn, graph=small)
        gbs = nbytes / (us * 1e-6) / 1e9
        kernels[name].update({"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                              "ms_per_step": round(us * kernels[name]["launches_per_step"] * 1e-3, 4)})
        if small:
            kernels[name]["timing"] = "CUDA-graph replay of the back-to-back calls (input resident in L2)"
    # The roofline is a single kernel's: the call with the largest share of the
    # step (its event-bracketed time in the step, which keeps what the step's
    # L2 state gives it) among those that are one kernel launch (the reducing
    # calls add a finalize, fp8_quantize_current is the amax kernel plus the
    # cast); its achieved bandwidth is that of its back-to-back launches.
    single = [k for k in kernels if k in SINGLE_KERNEL_CALLS and "us" in kernels[k]] or \
        [k for k in kernels if "us" in kernels[k]]
    dominant = max(single, key=lambda k: kernels[k]["bracketed_avg_us"] * kernels[k]["launches_per_step"])
    dk = kernels[dominant]
    traffic_per_elem = kernel_traffic(dominant)
    per_elem_bytes = {"quantize": 3, "quantize_delayed": 3, "quantize_grouped": 3, "cast_transpose": 4, "amax": 2,
                      "dequantize": 3}.get(dominant)
    alg_per_launch = dk["bytes_per_launch"]
    traffic = None
    if traffic_per_elem is not None and per_elem_bytes:
        traffic = round(traffic_per_elem * alg_per_launch / per_elem_bytes)
    cold_us = time_cold(back_to_back_calls(pipes, dev)[dominant][0], dev)
    value = world * step_bytes * args.steps / (ms_max * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME if full_suite else f"subset {','.join(which)} scale {args.scale} "
                                                                f"count {args.count or 'full'}",
                   "io": "bf16 in, e4m3/e5m2 uint8 codes out (W5: bf16 out)",
                   "bytes": "compulsory: each workload's inputs read once + outputs written once",
                   "compulsory_bytes_per_step": step_bytes, "kernel_bytes_per_step": kernel_bytes,
                   "kernel_gbs": round(world * kernel_bytes * args.steps / (ms_max * 1e-3) / 1e9, 1),
                   "l2": "no flush: inputs (%.2f GB) and per-step traffic (%.2f GB) exceed the 135 MB L2; every "
                         "W3 step and W5 tensor writes its own output buffers"
                         % (sum(t.numel() * t.element_size() for t in _all_inputs(inp)) / 1e9, kernel_bytes / 1e9),
                   "w5_path": "one grouped amax + scale call over the 32 tensors (per-tensor scales), then "
                              "per tensor its cast and its dequantize",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": dk["gbs"], "peak": peak, "unit": "GB/s",
                     "frac": round(dk["gbs"] / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": traffic, "algorithmic_bytes_per_launch": alg_per_launch,
                     "launch_us": dk["us"],
                     "timing": f"average of {B2B_LAUNCHES} back-to-back launches of the call on the launching "
                               f"stream (median of {B2B_GROUPS} groups), inputs cycled so that they exceed L2",
                     "bracketed_us": dk["bracketed_avg_us"],
                     "bracketed_frac": round(alg_per_launch / (dk["bracketed_avg_us"] * 1e-6) / 1e9 / peak, 4),
                     "cold_l2_us": round(cold_us, 2),
                     "cold_l2_timing": "mean of 20 single launches, the L2 flushed before each",
                     "cold_l2_frac": round(alg_per_launch / (cold_us * 1e-6) / 1e9 / peak, 4),
                     "dram_gbs": round(traffic / (dk["us"] * 1e-6) / 1e9, 1) if traffic else None},
        "kernels": kernels,
        "variants": variants,
        "kernel_timing": f"us/gbs/frac: {B2B_LAUNCHES} back-to-back launches between two events (median of "
                         f"{B2B_GROUPS} groups); bracketed_*: events around every launch of {ksteps} steps, which "
                         "adds each launch's dispatch latency; variants: {ksteps} steps with events only at "
                         "workload boundaries".replace("{ksteps}", str(ksteps)),
        "gpu_launches": launches,
        "clocks": clk,
    }
    if full_suite:
        result["config"]["inputs_sha256"] = input_digests(inp)
    if full_suite and not args.no_extras:
        result["extras"] = run_extras(inp, peak)
        result["extras_timing"] = EXTRAS_TIMING
    if not args.no_e2e and full_suite:
        del pipes
        torch.cuda.empty_cache()
        result["e2e"] = run_e2e(args, inp, step_bytes, world)
    if not args.no_cpu_baseline and rank == 0 and world == 1 and full_suite:
        result["cpu_baseline"], result["parity"] = cpu_baseline(args, inp, snap)
    else:
        result["parity"] = {"checked": False, "why": "the oracle runs only in the full-suite CPU baseline on rank 0"}
    return result


B2B_LAUNCHES, B2B_GROUPS = 20, 5


def back_to_back_calls(pipes, dev):
    """name -> (fn, algorithmic bytes per launch) for each call of the step.
    Each fn(i) issues the i-th of a run of identical launches; inputs cycle
    over distinct tensors wherever a workload has several, and the outputs of
    the W3 / W5 calls cycle over several buffers, so that consecutive launches
    neither read inputs nor overwrite outputs that are still in L2."""
    import torch
    import fp8_scaled_quantization_gb300 as fq
    calls = {}
    if "W1" in pipes:
        p = pipes["W1"]
        calls["quantize_current"] = (lambda i: fq.fp8_quantize_current(p.x, p.fmt, p.q, p.margin, p.amax, p.scale,
                                                                       p.scale_inv), p.bytes().total)
    if "W2" in pipes:
        p2 = pipes["W2"]
        b = p2.bytes().per_kernel
        calls["amax"] = (lambda i: fq.fp8_amax(p2.x, p2.amax, p2.fmt, p2.margin, p2.scale, p2.scale_inv),
                         b["amax"][0])
        calls["cast_transpose"] = (lambda i: fq.fp8_quantize_cast_transpose(p2.x, p2.fmt, p2.scale, p2.q_row,
                                                                            p2.q_col), b["cast_transpose"][0])
    if "W3" in pipes:
        p3 = pipes["W3"]
        q3 = [p3.q[0]] + [torch.empty_like(p3.q[0]) for _ in range(3)]
        calls["quantize_delayed"] = (lambda i, m=len(p3.xs): fq.fp8_quantize_delayed(
            p3.xs[i % m], p3.fmt, p3.scale, p3.scale_inv, q3[i % 4], p3.hist, i + 1, p3.algo, p3.margin,
            p3.amax[i % m:i % m + 1], p3.sat[i % m:i % m + 1]),
            p3.xs[0].numel() * (p3.xs[0].element_size() + 1) + p3.hist.numel() * 4 + 12)
        calls["update_delayed"] = (lambda i: fq.fp8_update_scale_delayed(p3.hist, i + 1, p3.amax[0:1], p3.algo, p3.fmt,
                                                                         p3.margin, p3.scale, p3.scale_inv),
                                   p3.hist.numel() * 4 + 12)
    if "W4" in pipes:
        p4 = pipes["W4"]
        b = p4.bytes().per_kernel
        calls["block128x128"] = (lambda i: fq.fp8_quantize_block(p4.w, 128, 128, p4.fmt, p4.q_w, p4.si_w),
                                 b["block128x128"][0])
        calls["block1x128"] = (lambda i: fq.fp8_quantize_block(p4.a, 1, 128, p4.fmt, p4.q_a, p4.si_a),
                               b["block1x128"][0])
    if "W5" in pipes:
        p5 = pipes["W5"]
        n5 = p5.xs[0].numel()
        calls["amax_grouped"] = (lambda i: fq.fp8_amax_grouped(p5.xs, p5.amax, p5.fmt, p5.margin, p5.scale,
                                                               p5.scale_inv),
                                 sum(x.numel() * x.element_size() for x in p5.xs))
        qs = [p5.q[0]] + [p5.q[0].clone() for _ in range(2)]
        ys = [p5.y[0], torch.empty_like(p5.y[0])]
        calls["quantize"] = (lambda i, m=len(p5.xs): fq.fp8_quantize(p5.xs[i % m], p5.fmt, p5.scale[i % m:i % m + 1],
                                                                     qs[i % 3]), n5 * 3)
        calls["dequantize"] = (lambda i: fq.fp8_dequantize(qs[i % 3], p5.fmt, p5.scale_inv[0:1], ys[i % 2]), n5 * 3)
    return calls


# Calls that move less than this are issued faster by the GPU than by the
# Python binding: their back-to-back launches are replayed from a CUDA graph.
B2B_GRAPH_BELOW_BYTES = 16 << 20


def time_back_to_back(fn, graph=False):
    """Average per-launch time (us) of B2B_LAUNCHES back-to-back calls, median
    of B2B_GROUPS groups; with `graph`, the calls are captured once in a CUDA
    graph on a side stream and the graph is replayed (GPU time, not the host's
    launch rate)."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per = []
    if graph:
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            for i in range(3):
                fn(i)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for i in range(B2B_LAUNCHES):
                    fn(i)
            g.replay()
            st.synchronize()
            for _ in range(B2B_GROUPS):
                e0.record(st)
                g.replay()
                e1.record(st)
                st.synchronize()
                per.append(e0.elapsed_time(e1) * 1e3 / B2B_LAUNCHES)
        torch.cuda.current_stream().wait_stream(st)
        return statistics.median(per)
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    for g in range(B2B_GROUPS):
        e0.record()
        for i in range(B2B_LAUNCHES):
            fn(g * B2B_LAUNCHES + i)
        e1.record()
        torch.cuda.synchronize()
        per.append(e0.elapsed_time(e1) * 1e3 / B2B_LAUNCHES)
    return statistics.median(per)


def flush_buffers(dev):
    import torch
    return (torch.empty(256 * 2 ** 20 // 4, dtype=torch.float32, device=dev),
            torch.ones(256 * 2 ** 20 // 4, dtype=torch.float32, device=dev))


def time_flushed(fn, dev, reps=20, bufs=None):
    """One call at a time between two events, the L2 flushed before every rep
    (EXTRAS_TIMING); returns (median, min, max, mean) in us over `reps` reps."""
    import torch
    flush, clean = bufs or flush_buffers(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for r in range(reps + 2):
        flush.fill_(float(r))
        clean.amax()
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        if r >= 2:
            ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts), min(ts), max(ts), statistics.mean(ts)


def time_cold(fn, dev):
    """Mean over 20 single launches with the L2 flushed before each (the event
    clock's 2.05 us steps make a median of single launches move in whole steps)."""
    return time_flushed(lambda: fn(0), dev)[3]


def _np(t):
    import numpy as np
    h = t.detach().contiguous().cpu()
    if h.dtype == __import__("torch").bfloat16:
        return h.view(__import__("torch").int16).numpy().view(np.uint16)
    return h.numpy()


def snapshot_outputs(pipes):
    """Host copies of what the last step left in each workload's outputs:
    W1/W2/W4 every output; W3 the last step's codes, every step's amax and
    saturation count, the history and the final scale; W5 the codes and the
    dequantized values of tensor 0 (the last one the step runs) and every
    tensor's amax and scales."""
    import numpy as np
    snap = {}
    if "W1" in pipes:
        p = pipes["W1"]
        snap["W1"] = {"q": _np(p.q), "amax": _np(p.amax), "scale": _np(p.scale), "scale_inv": _np(p.scale_inv)}
    if "W2" in pipes:
        p = pipes["W2"]
        snap["W2"] = {"q_row": _np(p.q_row), "q_col": _np(p.q_col), "amax": _np(p.amax), "scale": _np(p.scale),
                      "scale_inv": _np(p.scale_inv)}
    if "W3" in pipes:
        p = pipes["W3"]
        snap["W3"] = {"q_last": _np(p.q[-1]), "amax": _np(p.amax), "sat": _np(p.sat).astype(np.uint64),
                      "hist": _np(p.hist), "scale": _np(p.scale), "scale_inv": _np(p.scale_inv)}
    if "W4" in pipes:
        p = pipes["W4"]
        snap["W4"] = {"q_w": _np(p.q_w), "si_w": _np(p.si_w), "q_a": _np(p.q_a), "si_a": _np(p.si_a)}
    if "W5" in pipes:
        p = pipes["W5"]
        snap["W5"] = {"q0": _np(p.q[0]), "y0": _np(p.y[0]), "amax": _np(p.amax), "scale": _np(p.scale),
                      "scale_inv": _np(p.scale_inv)}
    return snap


def compare_parity(snap, ref):
    """Bit-for-bit comparison of the step's outputs with the oracle's, per workload."""
    import numpy as np
    out = {"checked": True}
    for w in ("W1", "W2", "W3", "W4", "W5"):
        if w not in snap or w not in ref:
            out[w] = "not checked"
            continue
        bad = []
        for k, want in ref[w].items():
            got = snap[w].get(k)
            want = np.asarray(want)
            if got is None or got.size != want.size or got.tobytes() != np.ascontiguousarray(
                    want.astype(got.dtype, copy=False)).tobytes():
                bad.append(k)
        out[w] = "bit-exact" if not bad else "MISMATCH: " + ", ".join(bad)
    out["what"] = ("the outputs of the last step run (W1, W2, W4 every output; W3 the codes of step 16, all "
                   "16 amax / saturation counts, the history and the final scale; W5 tensor 0's codes and "
                   "dequantized BF16 and all 32 amax / scale / scale_inv) against the oracle on the same bytes")
    return out


EXTRAS_TIMING = ("CUDA events around each call on the launching stream; before every rep (outside the "
                 "events) a 256 MB buffer is rewritten and then a second 256 MB buffer is read, so the inputs "
                 "are out of L2 and the flush's dirty lines are written back before the timed call; one "
                 "launch between two events reads in steps of about 2.05 us on these GPUs, so the median "
                 "moves by whole steps and the mean resolves below one")


def run_extras(inp, peak, reps=20):
    """Kernels beyond the five workloads, each timed on its own (EXTRAS_TIMING),
    median of `reps` reps with min, max and mean.  The read after the rewrite
    matters: a rewrite alone leaves the L2 full of dirty lines, and the timed
    kernel would pay for writing them back."""
    import torch
    import fp8_scaled_quantization_gb300 as fq
    dev = inp["w2"].device
    bufs = flush_buffers(dev)

    def timed(fn):
        return time_flushed(fn, dev, reps, bufs)

    def row(t, nbytes, what):
        us, lo, hi, mean = t if isinstance(t, tuple) else (t, None, None, None)
        gbs = nbytes / (us * 1e-6) / 1e9
        r = {"what": what, "us": round(us, 2), "bytes": int(nbytes), "gbs": round(gbs, 1),
             "frac": round(gbs / peak, 4)}
        if lo is not None:
            r.update({"median_us": round(us, 2), "min_us": round(lo, 2), "max_us": round(hi, 2),
                      "mean_us": round(mean, 2), "mean_frac": round(nbytes / (mean * 1e-6) / 1e9 / peak, 4),
                      "reps": reps})
        return r

    out = {}
    x = inp["w2"]
    r_, c_ = x.shape
    n = x.numel()
    qr = torch.empty((r_, c_), dtype=torch.uint8, device=dev)
    sr = torch.empty((r_, c_ // 32), dtype=torch.uint8, device=dev)
    qc = torch.empty((c_, r_), dtype=torch.uint8, device=dev)
    sc = torch.empty((c_, r_ // 32), dtype=torch.uint8, device=dev)
    us = timed(lambda: fq.fp8_quantize_mx(x, fq.E4M3, qr, sr, qc, sc))
    out["mx_quantize_rowwise_columnwise"] = row(us, n * 2 + 2 * (n + n // 32),
                                                "MXFP8 E4M3 1x32 + 32x1 (transposed), 8192x8192 BF16")
    y = torch.empty((r_, c_), dtype=torch.bfloat16, device=dev)
    us = timed(lambda: fq.fp8_dequantize_mx(qr, sr, fq.E4M3, y))
    out["mx_dequantize"] = row(us, n + n // 32 + 2 * n, "MXFP8 E4M3 -> BF16, 8192x8192")
    s_row = torch.full((1,), 300.0, device=dev)
    s_col = torch.full((1,), 2.0, device=dev)
    for src, key in ((fq.COLUMNWISE_FROM_ORIGINAL, "hybrid_from_original"),
                     (fq.COLUMNWISE_FROM_ROWWISE_DEQUANTIZED, "hybrid_from_rowwise_dequantized")):
        us = timed(lambda: fq.fp8_quantize_hybrid(x, fq.E4M3, s_row, qr, fq.E5M2, s_col, qc, src))
        out[key] = row(us, n * 2 + 2 * n, "rowwise E4M3 + columnwise E5M2 (transposed), 8192x8192 BF16")
    del qr, sr, qc, sc, y
    a = inp["w4"][1]
    ar, ac = a.shape
    na = a.numel()
    qr = torch.empty((ar, ac), dtype=torch.uint8, device=dev)
    sr = torch.empty((ar, ac // 128), dtype=torch.float32, device=dev)
    qc = torch.empty((ac, ar), dtype=torch.uint8, device=dev)
    sc = torch.empty((ac, ar // 128), dtype=torch.float32, device=dev)
    us = timed(lambda: fq.fp8_quantize_block_cast_transpose(a, fq.E4M3, qr, sr, qc, sc))
    out["block_cast_transpose"] = row(us, na * 2 + 2 * (na + 4 * na // 128),
                                      "E4M3 1x128 rowwise + 128x1 columnwise (transposed), 16384x7168 BF16")
    del qr, sr, qc, sc
    # FP32 inputs (master weights): the cast and current scaling of 8192 x 4096 fp32
    xf = inp["w2"][:, :4096].float().contiguous()
    nf = xf.numel()
    qf = torch.empty(xf.shape, dtype=torch.uint8, device=dev)
    sf = torch.full((1,), 0.25, device=dev)
    af, sif = torch.empty(1, device=dev), torch.empty(1, device=dev)
    out["fp32_quantize"] = row(timed(lambda: fq.fp8_quantize(xf, fq.E4M3, sf, qf)), nf * 5,
                               "FP32 8192x4096 -> E4M3 codes, given scale")
    out["fp32_current_scaling"] = row(timed(lambda: fq.fp8_quantize_current(xf, fq.E4M3, qf, 0, af, sf, sif)),
                                      nf * 5, "FP32 8192x4096 current scaling (amax + finalize + cast); "
                                      "compulsory 5 B/element")
    del xf, qf
    # W1 (1024 x 1024, 2 MB) is launch- and L2-bound: 20 current-scaling calls
    # captured in one CUDA graph, replayed with a warm L2
    x1 = inp["w1"]
    q1 = torch.empty(x1.shape, dtype=torch.uint8, device=dev)
    a1, s1, si1 = (torch.empty(1, device=dev) for _ in range(3))
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        fq.fp8_quantize_current(x1, fq.E4M3, q1, 0, a1, s1, si1)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            for _ in range(20):
                fq.fp8_quantize_current(x1, fq.E4M3, q1, 0, a1, s1, si1)
        graph.replay()
    st.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(10):
            graph.replay()
        e1.record(st)
    st.synchronize()
    us = e0.elapsed_time(e1) / 200 * 1e3
    out["w1_graph_warm_l2"] = row(us, x1.numel() * 3, "W1 current scaling (fp8_quantize_current), 20 calls per "
                                  "CUDA graph, warm L2; compulsory 3 B/element")
    # W1 as it runs in the step: issued right behind a large kernel, so its
    # launch overlaps that kernel's tail and its input is out of L2; the time
    # of (large kernel + W1) minus that of the large kernel alone, means of 60
    # (the event clock reads in steps of about 2.05 us, which a median keeps
    # and a mean resolves), the two kinds of rep interleaved
    big = torch.empty(64 << 20, dtype=torch.float32, device=dev)

    def pair_times():
        ts = {True: [], False: []}
        for r in range(124):
            with_w1 = bool(r & 1)
            e0.record()
            big.mul_(1.0)
            if with_w1:
                fq.fp8_quantize_current(x1, fq.E4M3, q1, 0, a1, s1, si1)
            e1.record()
            torch.cuda.synchronize()
            if r >= 4:
                ts[with_w1].append(e0.elapsed_time(e1) * 1e3)
        return statistics.mean(ts[True]), statistics.mean(ts[False])

    with_w1_us, without_us = pair_times()
    us = with_w1_us - without_us
    out["w1_behind_large_kernel"] = row(us, x1.numel() * 3, "W1 current scaling issued right behind a 256 MB "
                                        "kernel (launch overlapped, input out of L2): (kernel + W1) - kernel, "
                                        "means of 60, interleaved; compulsory 3 B/element")
    del big
    del q1
    # 64 expert-sized tensors: grouped current scaling vs per-tensor calls
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    rows = torch.randint(128, 2048, (64,), generator=g, device=dev).tolist()
    xs = [torch.randn((int(rr), 7168), generator=g, device=dev).to(torch.bfloat16) for rr in rows]
    qs = [torch.empty(t.shape, dtype=torch.uint8, device=dev) for t in xs]
    m = len(xs)
    am, s_, si_ = (torch.empty(m, device=dev) for _ in range(3))
    nbytes = sum(t.numel() * 3 for t in xs)

    def grouped():
        fq.fp8_amax_grouped(xs, am, fq.E4M3, 0, s_, si_)
        fq.fp8_quantize_grouped(xs, fq.E4M3, s_, qs)

    def per_tensor():
        for i, t in enumerate(xs):
            fq.fp8_amax(t, am[i:i + 1], fq.E4M3, 0, s_[i:i + 1], si_[i:i + 1])
            fq.fp8_quantize(t, fq.E4M3, s_[i:i + 1], qs[i])

    out["grouped_current_scaling"] = row(timed(grouped), nbytes,
                                         "64 BF16 tensors [128..2047, 7168]: amax+scale+cast, grouped (3 launches)")
    out["per_tensor_current_scaling"] = row(timed(per_tensor), nbytes,
                                            "the same 64 tensors, per-tensor calls (192 launches)")
    del xs, qs
    # The 32 W5 gradient tensors: grouped current scaling vs the per-tensor call
    if len(inp.get("w5", [])) > 1:
        x5 = inp["w5"]
        q5 = [torch.empty(t.shape, dtype=torch.uint8, device=dev) for t in x5]
        a5, s5, si5 = (torch.empty(len(x5), device=dev) for _ in range(3))

        def grouped5():
            fq.fp8_amax_grouped(x5, a5, fq.E5M2, 0, s5, si5)
            fq.fp8_quantize_grouped(x5, fq.E5M2, s5, q5)

        def per_tensor5():
            for i, t in enumerate(x5):
                fq.fp8_quantize_current(t, fq.E5M2, q5[i], 0, a5[i:i + 1], s5[i:i + 1], si5[i:i + 1])

        nb5 = sum(t.numel() * 5 for t in x5)
        out["w5_grouped_current_scaling"] = row(timed(grouped5), nb5, f"the {len(x5)} W5 tensors (8192x8192 BF16, "
                                                "E5M2): amax+scale+cast grouped (3 launches); 5 B/element")
        out["w5_per_tensor_current_scaling"] = row(timed(per_tensor5), nb5, f"the same {len(x5)} tensors, "
                                                   "fp8_quantize_current per tensor; 5 B/element")
        del q5
    # FP32 master-weight shards: 32 tensors [512..1535, 4096] fp32, grouped
    rows32 = torch.randint(512, 1536, (32,), generator=g, device=dev).tolist()
    ws32 = [torch.randn((int(rr), 4096), generator=g, device=dev) for rr in rows32]
    qs32 = [torch.empty(t.shape, dtype=torch.uint8, device=dev) for t in ws32]
    a32, s32, si32 = (torch.empty(32, device=dev) for _ in range(3))

    def grouped32():
        fq.fp8_amax_grouped(ws32, a32, fq.E4M3, 0, s32, si32)
        fq.fp8_quantize_grouped(ws32, fq.E4M3, s32, qs32)

    out["grouped_fp32_master_weights"] = row(timed(grouped32), sum(t.numel() * 5 for t in ws32),
                                             "32 FP32 tensors [512..1535, 4096]: amax+scale+cast, grouped")
    return out


def run_extras_only(args):
    import torch
    import fp8_scaled_quantization_gb300 as fq
    fq.library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    inp = make_inputs(workload_shapes(1.0), dev, which=("W1", "W2", "W4"))
    peak, _ = measured_hbm_peak()
    return {"metric": METRIC, "unit": UNIT, "extras": run_extras(inp, peak, reps=max(1, args.steps)),
            "extras_timing": EXTRAS_TIMING}


def input_digests(inp):
    """SHA-256 of each workload's input bytes (tensors in generation order), first 16 hex digits."""
    out = {}
    for key in ("w1", "w2", "w3", "w4", "w5"):
        v = inp[key]
        tensors = v if isinstance(v, (list, tuple)) else [v]
        h = hashlib.sha256()
        for t in tensors:
            h.update(t.detach().contiguous().view(-1).view(torch_uint8()).cpu().numpy().tobytes())
        out[key.upper()] = h.hexdigest()[:16]
    return out


def torch_uint8():
    import torch
    return torch.uint8


def _all_inputs(inp):
    out = []
    for k in ("w1", "w2"):
        if k in inp:
            out.append(inp[k])
    for k in ("w3", "w4", "w5"):
        if k in inp:
            out.extend(inp[k])
    return out


def run_e2e(args, inp, step_bytes, world):
    """The same step through the public API with host buffers: every step
    copies each workload's inputs host->device from pinned memory and reads
    its results (codes and scales; W5: the dequantized BF16) back.  Copies in,
    kernels and copies out run on three streams, one item (tensor or step)
    at a time, ordered by events, with separate device outputs per item."""
    import torch
    from fp8_scaled_quantization_gb300 import pipelines as P, E4M3, E5M2
    p1 = P.CurrentScaling(inp["w1"], E4M3, 0)
    p2 = P.CurrentCastTranspose(inp["w2"], E4M3, 1)
    p3 = P.DelayedScaling(inp["w3"], 1024, E4M3, 0, keep_codes=True)
    p4 = P.BlockScaling(*inp["w4"], E4M3)
    p5 = P.GradientQDQ(inp["w5"], E5M2, 0, keep_outputs=True)
    items = [([p1.x], p1.run, [p1.q, p1.scale_inv]),
             ([p2.x], p2.run, [p2.q_row, p2.q_col, p2.scale_inv])]
    for k in range(len(p3.xs)):
        last = [p3.amax, p3.sat, p3.scale_inv] if k == len(p3.xs) - 1 else []
        items.append(([p3.xs[k]], (lambda k=k: p3.run_step(k)), [p3.q[k]] + last))
    items.append((list(inp["w4"]), p4.run, [p4.q_w, p4.si_w, p4.q_a, p4.si_a]))
    for k in range(len(p5.xs)):
        last = [p5.scale_inv] if k == len(p5.xs) - 1 else []
        items.append(([p5.xs[k]], (lambda k=k: p5.run_tensor(k)), [p5.y[k]] + last))
    h_in = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in ins] for ins, _, _ in items]
    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs] for _, _, outs in items]
    h2d = sum(t.numel() * t.element_size() for v in h_in for t in v)
    d2h = sum(t.numel() * t.element_size() for v in h_out for t in v)
    s_comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    prev_comp, prev_out = [None] * len(items), [None] * len(items)

    def e2e_step():
        for i, (ins, fn, outs) in enumerate(items):
            with torch.cuda.stream(s_in):
                if prev_comp[i] is not None:
                    s_in.wait_event(prev_comp[i])  # the last step's kernels are done with these inputs
                for h, d in zip(h_in[i], ins):
                    d.copy_(h, non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(s_in)
            s_comp.wait_event(e_in)
            if prev_out[i] is not None:
                s_comp.wait_event(prev_out[i])  # the last step's results have been read back
            fn()
            e_c = torch.cuda.Event()
            e_c.record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_c)
                for h, d in zip(h_out[i], outs):
                    h.copy_(d, non_blocking=True)
                e_o = torch.cuda.Event()
                e_o.record(s_out)
            prev_comp[i], prev_out[i] = e_c, e_o

    steps = max(1, min(args.steps, 5))
    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t = time.perf_counter()
    for _ in range(steps):
        e2e_step()
    torch.cuda.synchronize()
    dt = max_over_ranks((time.perf_counter() - t) * 1e3, world)
    return {"value": round(world * step_bytes * steps / (dt * 1e-3) / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(dt / steps, 3),
            "note": "pinned host buffers; copies in, kernels and copies out overlapped on three streams"}


# --------------------------------------------------------------- CPU oracle

def oracle_suite_sample(inp_host, fraction, threads, collect=None):
    """Run the oracle over a sample of every workload; returns algorithmic bytes.
    With a dict `collect`, keep the outputs that snapshot_outputs() keeps of
    the GPU's step (keeping them is a reference, not work)."""
    import numpy as np
    import oracle as O

    def rows(x, f):
        r = max(1, int(x.shape[0] * f))
        return np.ascontiguousarray(x[:r])

    c = collect if collect is not None else {}
    nbytes = 0
    x1 = inp_host["w1"]
    a1 = O.amax(x1, threads)
    s, si = O.compute_scale(a1, O.E4M3, 0)
    q1, _ = O.quantize(x1, O.E4M3, s, threads)
    c["W1"] = {"q": q1, "amax": np.float32(a1), "scale": s, "scale_inv": si}
    nbytes += x1.size * 5
    x2 = rows(inp_host["w2"], fraction)
    a2 = O.amax(x2, threads)
    s, si = O.compute_scale(a2, O.E4M3, 1)
    qr, qc = O.cast_transpose(x2, O.E4M3, s, threads)
    c["W2"] = {"q_row": qr, "q_col": qc, "amax": np.float32(a2), "scale": s, "scale_inv": si}
    nbytes += x2.size * 6
    hist = np.zeros(1024, np.float32)
    s, si = O.update_delayed(hist, 0, None, O.ALGO_MAX, O.E4M3, 0)
    am3, sat3, q3 = [], [], None
    for k, x in enumerate(inp_host["w3"]):
        x = rows(x, fraction)
        q3, sat = O.quantize(x, O.E4M3, s, threads)
        a = O.amax(x, threads)
        s, si = O.update_delayed(hist, k, a, O.ALGO_MAX, O.E4M3, 0)
        am3.append(a)
        sat3.append(sat)
        nbytes += x.size * 3
    c["W3"] = {"q_last": q3, "amax": np.array(am3, np.float32), "sat": np.array(sat3, np.uint64), "hist": hist,
               "scale": s, "scale_inv": si}
    w, a = inp_host["w4"]
    w = rows(w, fraction)
    w = w[: max(128, w.shape[0] // 128 * 128)]
    qw, siw = O.quantize_block(np.ascontiguousarray(w), 128, 128, O.E4M3, threads)
    a = rows(a, fraction)
    qa, sia = O.quantize_block(a, 1, 128, O.E4M3, threads)
    c["W4"] = {"q_w": qw, "si_w": siw, "q_a": qa, "si_a": sia}
    nbytes += w.size * 3 + a.size * 3
    am5, s5, si5 = [], [], []
    for k, x in enumerate(inp_host["w5"]):
        x = rows(x, fraction)
        a = O.amax(x, threads)
        s, si = O.compute_scale(a, O.E5M2, 0)
        q, _ = O.quantize(x, O.E5M2, s, threads)
        y = O.dequantize(q, O.E5M2, np.array([si], np.float32), threads=threads)
        am5.append(a)
        s5.append(s)
        si5.append(si)
        if k == 0:
            c["W5"] = {"q0": q, "y0": y}
        nbytes += x.size * 8
    c["W5"].update({"amax": np.array(am5, np.float32), "scale": np.array(s5, np.float32),
                    "scale_inv": np.array(si5, np.float32)})
    return nbytes


def host_sample(inp, fraction, max_w3=4, max_w5=4):
    """Host copies of the leading rows of each workload tensor (a bounded sample)."""
    from fp8_scaled_quantization_gb300.workloads import bf16_bits

    def r(x):
        return bf16_bits(x[: max(1, int(x.shape[0] * fraction))])

    return {"w1": bf16_bits(inp["w1"]), "w2": r(inp["w2"]), "w3": [r(x) for x in inp["w3"][:max_w3]],
            "w4": (r(inp["w4"][0]), r(inp["w4"][1])), "w5": [r(x) for x in inp["w5"][:max_w5]]}


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(args, inp, snap=None):
    """The oracle as it stands over the workloads (timed), then -- outside the
    timing -- its outputs compared bit for bit with the GPU step's (`snap`).
    Returns (cpu_baseline, parity)."""
    import numpy as np
    import oracle as O
    O.build()
    sample = host_sample(inp, args.cpu_fraction, max_w3=len(inp["w3"]), max_w5=len(inp["w5"]))
    threads = cpu_threads()
    ref = {}
    t = time.perf_counter()
    nbytes = oracle_suite_sample(sample, 1.0, threads, ref)
    dt = time.perf_counter() - t
    if snap is None:
        parity = {"checked": False, "why": "no snapshot of the step's outputs"}
    elif args.cpu_fraction != 1.0:
        parity = {"checked": False, "why": "the CPU baseline ran on a row sample (--cpu-fraction)"}
    else:
        parity = compare_parity(snap, ref)
    del ref
    # single-threaded: W1 (amax, scale, cast), the oracle's own bytes
    x1 = sample["w1"]
    t1 = time.perf_counter()
    s1, _ = O.compute_scale(O.amax(x1, 1), O.E4M3, 0)
    O.quantize(x1, O.E4M3, s1, 1)
    dt1 = time.perf_counter() - t1
    # single-threaded: one W5 tensor (amax, scale, quantize, dequantize)
    x5 = sample["w5"][0]
    t5 = time.perf_counter()
    s5, si5 = O.compute_scale(O.amax(x5, 1), O.E5M2, 0)
    q5, _ = O.quantize(x5, O.E5M2, s5, 1)
    O.dequantize(q5, O.E5M2, np.array([si5], np.float32), threads=1)
    dt5 = time.perf_counter() - t5
    return ({"value": round(nbytes / dt / 1e9, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
             "seconds": round(dt, 2), "single_thread_w1_gbs": round(x1.size * 5 / dt1 / 1e9, 3),
             "single_thread_w5_tensor_gbs": round(x5.size * 8 / dt5 / 1e9, 3),
             "sample": f"leading {args.cpu_fraction:.4g} of the rows of every tensor of W1-W5 (all 16 W3 steps, "
                       f"all 32 W5 tensors), one pass; the oracle's own algorithmic bytes ({nbytes / 1e9:.2f} GB)"},
            parity)


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on a bounded sample of each workload."""
    import oracle as O
    import torch
    from fp8_scaled_quantization_gb300 import workloads as wl
    O.build()
    shapes = workload_shapes(args.scale)
    f = 1.0 / 8
    shp = lambda s: (max(128, int(s[0] * f) // 128 * 128), s[1])  # noqa: E731
    inp = {"w1": wl.w1_outliers(shapes["w1"]), "w2": wl.w2_student_t(shp(shapes["w2"])),
           "w3": list(wl.w3_steps(shp(shapes["w3"]), 4)),
           "w4": wl.w4_block(shp(shapes["w4w"]), shp(shapes["w4a"])),
           "w5": list(wl.w5_gradients(shp(shapes["w5"]), 4))}
    sample = host_sample(inp, 1.0)
    threads = cpu_threads()
    torch.set_num_threads(max(1, threads))
    for _ in range(args.warmup):
        oracle_suite_sample(sample, 1.0, threads)
    t = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += oracle_suite_sample(sample, 1.0, threads)
    dt = time.perf_counter() - t
    v = round(nbytes / dt / 1e9, 3)
    desc = ("each step: the oracle on 1/8 of the rows of W2, of W4, of 4 of the 16 W3 steps and of 4 of the 32 "
            "W5 tensors, and on all of W1 (CPU-generated inputs of the same distributions)")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME, "sample": desc},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------- plumbing

def max_over_ranks(v: float, world: int) -> float:
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # the CPU oracle runs once, on rank 0; other ranks exit without work
        if rank == 0:
            print(json.dumps(run_reference(args, 0, world)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group(backend)
    if args.extras_only:
        if rank == 0:
            print(json.dumps(run_extras_only(args)), flush=True)
        return
    res = run_ours(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
