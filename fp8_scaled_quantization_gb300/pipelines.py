"""The FP8 scaling recipes as preallocated launch sequences over the C ABI.

Each pipeline owns its device outputs, enqueues its kernels on the current
stream in ``run()`` and reports the algorithmic bytes one run moves (read
once + written once, per kernel).  Nothing here computes: every step is a
call into the CUDA library.

  CurrentScaling     "Megatron FP8" §4/§10: fp8_quantize_current (amax kernel, then a cast
                     that derives the scale itself), or fp8_amax (+ scale) -> fp8_quantize
  CurrentCastTranspose  same, with rowwise + columnwise outputs (§6)
  DelayedScaling     §5: per step fp8_quantize_delayed (the cast records amax and the
                     saturation count; its finalize writes the history ring and the next
                     scale), or fp8_quantize -> fp8_update_scale_delayed
  BlockScaling       "Low Precision Training and Rollout": fp8_quantize_block
                     128 x 128 (weight) and 1 x 128 (activation)
  GradientQDQ        E5M2 current scaling then fp8_dequantize back to BF16, per tensor or
                     with one grouped amax + scale call over all tensors (§21)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import (AMAX_MAX, E4M3, E5M2, fp8_amax, fp8_amax_grouped, fp8_dequantize, fp8_quantize, fp8_quantize_block,
               fp8_quantize_cast_transpose, fp8_quantize_current, fp8_quantize_delayed, fp8_quantize_grouped,
               fp8_update_scale_delayed)


def _f32(dev, n=1, fill=None):
    t = torch.empty(n, dtype=torch.float32, device=dev)
    if fill is not None:
        t.fill_(fill)
    return t


@dataclass
class KernelBytes:
    """Algorithmic bytes moved by each kernel of one run (name -> bytes per launch, launches)."""
    per_kernel: dict = field(default_factory=dict)

    def add(self, name: str, nbytes: int, launches: int = 1):
        b, n = self.per_kernel.get(name, (0, 0))
        self.per_kernel[name] = (b + nbytes * launches, n + launches)

    @property
    def total(self) -> int:
        return sum(b for b, _ in self.per_kernel.values())

    @property
    def launches(self) -> int:
        return sum(n for _, n in self.per_kernel.values())


def esize(x: torch.Tensor) -> int:
    return x.element_size()


class CurrentScaling:
    """Per-tensor current scaling: one fp8_quantize_current call (current_call=True),
    or fp8_amax (amax + scale) followed by fp8_quantize."""

    def __init__(self, x: torch.Tensor, fmt: int = E4M3, margin: int = 0, current_call: bool = True):
        self.x, self.fmt, self.margin, self.current_call = x, fmt, margin, current_call
        dev = x.device
        self.q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        self.amax, self.scale, self.scale_inv = _f32(dev), _f32(dev), _f32(dev)

    def run(self, timer=None):
        if self.current_call:
            _t(timer, "quantize_current", lambda: fp8_quantize_current(self.x, self.fmt, self.q, self.margin,
                                                                       self.amax, self.scale, self.scale_inv))
            return
        _t(timer, "amax", lambda: fp8_amax(self.x, self.amax, self.fmt, self.margin, self.scale, self.scale_inv))
        _t(timer, "quantize", lambda: fp8_quantize(self.x, self.fmt, self.scale, self.q))

    def bytes(self) -> KernelBytes:
        n, b = self.x.numel(), KernelBytes()
        if self.current_call:  # the amax kernel's read of x and the cast
            b.add("quantize_current", n * esize(self.x) + n * (esize(self.x) + 1))
            return b
        b.add("amax", n * esize(self.x))
        b.add("quantize", n * (esize(self.x) + 1))
        return b


class CurrentCastTranspose:
    """Current scaling with rowwise and columnwise (transposed) codes."""

    def __init__(self, x: torch.Tensor, fmt: int = E4M3, margin: int = 1):
        self.x, self.fmt, self.margin = x, fmt, margin
        dev = x.device
        r, c = x.shape
        self.q_row = torch.empty((r, c), dtype=torch.uint8, device=dev)
        self.q_col = torch.empty((c, r), dtype=torch.uint8, device=dev)
        self.amax, self.scale, self.scale_inv = _f32(dev), _f32(dev), _f32(dev)

    def run(self, timer=None):
        _t(timer, "amax", lambda: fp8_amax(self.x, self.amax, self.fmt, self.margin, self.scale, self.scale_inv))
        _t(timer, "cast_transpose",
           lambda: fp8_quantize_cast_transpose(self.x, self.fmt, self.scale, self.q_row, self.q_col))

    def bytes(self) -> KernelBytes:
        n, b = self.x.numel(), KernelBytes()
        b.add("amax", n * esize(self.x))
        b.add("cast_transpose", n * (esize(self.x) + 2))
        return b


class DelayedScaling:
    """Delayed scaling over a sequence of tensors sharing one amax history.

    A run starts from a zero history (scale 1 at step 0) and, per step k,
    casts x_k with the current scale while recording amax_k and the saturated
    count, then writes amax_k into slot k % len and derives the next scale.
    With fused=True (the default) each step is one fp8_quantize_delayed
    launch; fused=False issues fp8_quantize + fp8_update_scale_delayed."""

    def __init__(self, xs: list, history_len: int = 1024, fmt: int = E4M3, margin: int = 0,
                 algo: int = AMAX_MAX, keep_codes: bool = False, record_scales: bool = False,
                 fused: bool = True):
        self.xs, self.fmt, self.margin, self.algo, self.fused = xs, fmt, margin, algo, fused
        dev = xs[0].device
        self.hist = torch.zeros(history_len, dtype=torch.float32, device=dev)
        self.scale, self.scale_inv = _f32(dev), _f32(dev)
        self.amax = torch.empty(len(xs), dtype=torch.float32, device=dev)
        self.sat = torch.empty(len(xs), dtype=torch.int64, device=dev)
        # the scale used at each step (a device copy per step; for checking only)
        self.scales = torch.empty(len(xs), dtype=torch.float32, device=dev) if record_scales else None
        n = len(xs) if keep_codes else 1
        self.q = [torch.empty(xs[0].shape, dtype=torch.uint8, device=dev) for _ in range(n)]

    def run(self, timer=None):
        for k in range(len(self.xs)):
            self.run_step(k, timer)

    def run_step(self, k: int, timer=None):
        """Step k of the sequence (step 0 also resets the history and the scale)."""
        if k == 0:
            self.hist.zero_()
            _t(timer, "update_delayed", lambda: fp8_update_scale_delayed(self.hist, 0, None, self.algo, self.fmt,
                                                                         self.margin, self.scale, self.scale_inv))
        x, q = self.xs[k], self.q[k % len(self.q)]
        if self.scales is not None:
            self.scales[k:k + 1].copy_(self.scale)
        if self.fused:
            _t(timer, "quantize_delayed", lambda: fp8_quantize_delayed(
                x, self.fmt, self.scale, self.scale_inv, q, self.hist, k, self.algo, self.margin,
                self.amax[k:k + 1], self.sat[k:k + 1]))
            return
        _t(timer, "quantize", lambda: fp8_quantize(x, self.fmt, self.scale, q, self.amax[k:k + 1],
                                                   self.sat[k:k + 1]))
        _t(timer, "update_delayed", lambda: fp8_update_scale_delayed(
            self.hist, k, self.amax[k:k + 1], self.algo, self.fmt, self.margin, self.scale, self.scale_inv))

    def bytes(self) -> KernelBytes:
        b = KernelBytes()
        hist_bytes = self.hist.numel() * 4 + 4 + 8
        for x in self.xs:
            if self.fused:
                b.add("quantize_delayed", x.numel() * (esize(x) + 1) + hist_bytes)
            else:
                b.add("quantize", x.numel() * (esize(x) + 1))
        b.add("update_delayed", hist_bytes, 1 if self.fused else len(self.xs) + 1)
        return b


class BlockScaling:
    """128 x 128 block scales for a weight and 1 x 128 tile scales for an activation."""

    def __init__(self, weight: torch.Tensor, act: torch.Tensor, fmt: int = E4M3):
        self.w, self.a, self.fmt = weight, act, fmt
        dev = weight.device
        (wr, wc), (ar, ac) = weight.shape, act.shape
        self.q_w = torch.empty((wr, wc), dtype=torch.uint8, device=dev)
        self.si_w = torch.empty((-(-wr // 128), -(-wc // 128)), dtype=torch.float32, device=dev)
        self.q_a = torch.empty((ar, ac), dtype=torch.uint8, device=dev)
        self.si_a = torch.empty((ar, -(-ac // 128)), dtype=torch.float32, device=dev)

    def run(self, timer=None):
        _t(timer, "block128x128", lambda: fp8_quantize_block(self.w, 128, 128, self.fmt, self.q_w, self.si_w))
        _t(timer, "block1x128", lambda: fp8_quantize_block(self.a, 1, 128, self.fmt, self.q_a, self.si_a))

    def bytes(self) -> KernelBytes:
        b = KernelBytes()
        b.add("block128x128", self.w.numel() * (esize(self.w) + 1) + self.si_w.numel() * 4)
        b.add("block1x128", self.a.numel() * (esize(self.a) + 1) + self.si_a.numel() * 4)
        return b


class GradientQDQ:
    """Per tensor: E5M2 current scaling, then dequantize back to BF16.

    group="all": the amax, scale and cast of all tensors are two grouped calls
    (every tensor keeps its own amax and scale; three launches in all), then
    each tensor is dequantized, last tensor first, so that the codes written
    last are read while still in L2.  group="amax": one grouped amax + scale
    call for all tensors, then per tensor the cast and, right after it, the
    dequantize, which reads the codes while they are still in L2.  Otherwise
    (group="", and in run_tensor, which the host-buffer path uses one tensor
    at a time) each tensor is one fp8_quantize_current call (current_call=True)
    or fp8_amax + fp8_quantize, then its dequantize."""

    def __init__(self, xs: list, fmt: int = E5M2, margin: int = 0, keep_outputs: bool = False,
                 current_call: bool = True, group: str = ""):
        if group not in ("", "amax", "all"):
            raise ValueError("group must be '', 'amax' or 'all'")
        self.xs, self.fmt, self.margin, self.current_call, self.group = xs, fmt, margin, current_call, group
        dev = xs[0].device
        nq = len(xs) if (keep_outputs or group == "all") else 1  # the grouped cast writes every tensor's codes
        ny = len(xs) if keep_outputs else 1
        self.q = [torch.empty(xs[0].shape, dtype=torch.uint8, device=dev) for _ in range(nq)]
        self.y = [torch.empty(xs[0].shape, dtype=torch.bfloat16, device=dev) for _ in range(ny)]
        self.amax = torch.empty(len(xs), dtype=torch.float32, device=dev)
        self.scale = torch.empty(len(xs), dtype=torch.float32, device=dev)
        self.scale_inv = torch.empty(len(xs), dtype=torch.float32, device=dev)

    def run(self, timer=None):
        if not self.group:
            for k in range(len(self.xs)):
                self.run_tensor(k, timer)
            return
        _t(timer, "amax_grouped", lambda: fp8_amax_grouped(self.xs, self.amax, self.fmt, self.margin, self.scale,
                                                           self.scale_inv))
        if self.group == "amax":
            # last tensor first: the grouped amax read it last, so its tail is still in L2
            for k in reversed(range(len(self.xs))):
                x, q, y = self.xs[k], self.q[k % len(self.q)], self.y[k % len(self.y)]
                s, si = self.scale[k:k + 1], self.scale_inv[k:k + 1]
                _t(timer, "quantize", lambda: fp8_quantize(x, self.fmt, s, q))
                _t(timer, "dequantize", lambda: fp8_dequantize(q, self.fmt, si, y))
            return
        _t(timer, "quantize_grouped", lambda: fp8_quantize_grouped(self.xs, self.fmt, self.scale, self.q))
        for k in reversed(range(len(self.xs))):
            q, y, si = self.q[k], self.y[k % len(self.y)], self.scale_inv[k:k + 1]
            _t(timer, "dequantize", lambda: fp8_dequantize(q, self.fmt, si, y))

    def run_tensor(self, k: int, timer=None):
        x, q, y = self.xs[k], self.q[k % len(self.q)], self.y[k % len(self.y)]
        s, si = self.scale[k:k + 1], self.scale_inv[k:k + 1]
        if self.current_call:
            _t(timer, "quantize_current",
               lambda: fp8_quantize_current(x, self.fmt, q, self.margin, self.amax[k:k + 1], s, si))
        else:
            _t(timer, "amax", lambda: fp8_amax(x, self.amax[k:k + 1], self.fmt, self.margin, s, si))
            _t(timer, "quantize", lambda: fp8_quantize(x, self.fmt, s, q))
        _t(timer, "dequantize", lambda: fp8_dequantize(q, self.fmt, si, y))

    def bytes(self) -> KernelBytes:
        b = KernelBytes()
        if self.group:
            b.add("amax_grouped", sum(x.numel() * esize(x) for x in self.xs))
            if self.group == "all":
                b.add("quantize_grouped", sum(x.numel() * (esize(x) + 1) for x in self.xs))
            for x in self.xs:
                if self.group == "amax":
                    b.add("quantize", x.numel() * (esize(x) + 1))
                b.add("dequantize", x.numel() * (1 + 2))
            return b
        for x in self.xs:
            n = x.numel()
            if self.current_call:
                b.add("quantize_current", n * esize(x) + n * (esize(x) + 1))
            else:
                b.add("amax", n * esize(x))
                b.add("quantize", n * (esize(x) + 1))
            b.add("dequantize", n * (1 + 2))
        return b


def _t(timer, name, fn):
    """Run `fn`, bracketed by the timer's events for kernel `name` when a timer is given."""
    if timer is None:
        fn()
    else:
        timer.start(name)
        fn()
        timer.stop(name)
