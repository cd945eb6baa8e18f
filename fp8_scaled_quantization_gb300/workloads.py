"""Seeded synthetic inputs shaped like the transformer tensors the FP8 recipes
quantize.  This module only draws random numbers; it holds none of the
quantization arithmetic, and both the CUDA path and the CPU oracle consume the
same bytes it produces (the oracle through a host copy).

The five workloads (sizes are the defaults; tests pass smaller shapes):
  W1  per-tensor current scaling, E4M3, margin 0: one BF16 [1024, 1024],
      N(0,1) * 64 with 16 entries at random positions set to +-2000.
  W2  current-scaling cast + transpose, E4M3, margin 1: BF16 [8192, 8192],
      Student-t(nu=3) * 4.
  W3  delayed scaling, E4M3, history 1024, algo max, margin 0: 16 steps of
      BF16 [4096, 14336], N(0,1) * 8 * 1.1^k at step k.
  W4  blockwise E4M3: weight BF16 [7168, 18432] with one lognormal(0, 2)
      magnitude per 128 x 128 block times N(0,1); activation BF16
      [16384, 7168] with one lognormal(0, 2) magnitude per 1 x 128 tile
      times N(0,1) (same generator, drawn after the weight).
  W5  E5M2 gradients: 32 BF16 [8192, 8192], Laplace(0, 1e-3), 10 % exact
      zeros, 0.01 % of entries multiplied by 1e4; current scaling, then
      dequantize back to BF16.

Values are drawn in fp32 with a ``torch.Generator`` on the requested device
and rounded to BF16 (round to nearest even).  The bytes depend on the device
of the generator; parity always hands the same bytes to both sides.
"""
from __future__ import annotations

import torch

SEEDS = {"w1": 0, "w2": 1, "w3": 2, "w4": 3, "w5": 4}

W1_SHAPE = (1024, 1024)
W2_SHAPE = (8192, 8192)
W3_SHAPE, W3_STEPS, W3_HISTORY = (4096, 14336), 16, 1024
W4_WEIGHT_SHAPE, W4_ACT_SHAPE = (7168, 18432), (16384, 7168)
W5_SHAPE, W5_TENSORS = (8192, 8192), 32


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def w1_outliers(shape=W1_SHAPE, device="cpu", n_outliers=16, seed=SEEDS["w1"]) -> torch.Tensor:
    g = generator(seed, device)
    x = _randn(shape, g, device) * 64.0
    flat = x.view(-1)
    k = min(n_outliers, flat.numel())
    pos = torch.randperm(flat.numel(), generator=g, device=device)[:k]
    sign = torch.randint(0, 2, (k,), generator=g, device=device).to(torch.float32) * 2.0 - 1.0
    flat[pos] = 2000.0 * sign
    return x.to(torch.bfloat16)


def w2_student_t(shape=W2_SHAPE, device="cpu", seed=SEEDS["w2"], nu: int = 3) -> torch.Tensor:
    g = generator(seed, device)
    z = _randn(shape, g, device)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(nu):
        chi2 += _randn(shape, g, device) ** 2
    return (z / torch.sqrt(chi2 / nu) * 4.0).to(torch.bfloat16)


def w3_steps(shape=W3_SHAPE, steps=W3_STEPS, device="cpu", seed=SEEDS["w3"]):
    """Yields the BF16 tensor of each step k = 0 .. steps-1."""
    g = generator(seed, device)
    for k in range(steps):
        yield (_randn(shape, g, device) * (8.0 * 1.1 ** k)).to(torch.bfloat16)


def _block_magnitudes(rows, cols, br, bc, g, device):
    nbr, nbc = -(-rows // br), -(-cols // bc)
    mag = torch.exp(2.0 * _randn((nbr, nbc), g, device))  # lognormal(mu=0, sigma=2)
    return mag.repeat_interleave(br, 0)[:rows].repeat_interleave(bc, 1)[:, :cols]


def w4_block(weight_shape=W4_WEIGHT_SHAPE, act_shape=W4_ACT_SHAPE, device="cpu", seed=SEEDS["w4"]):
    """(weight with per-128x128 magnitudes, activation with per-1x128 magnitudes)."""
    g = generator(seed, device)
    wm = _block_magnitudes(*weight_shape, 128, 128, g, device)
    w = (_randn(weight_shape, g, device) * wm).to(torch.bfloat16)
    del wm
    am = _block_magnitudes(*act_shape, 1, 128, g, device)
    a = (_randn(act_shape, g, device) * am).to(torch.bfloat16)
    return w, a


def w5_gradients(shape=W5_SHAPE, count=W5_TENSORS, device="cpu", seed=SEEDS["w5"], scale=1e-3,
                 zero_frac=0.10, spike_frac=1e-4, spike=1e4):
    """Yields `count` BF16 gradient-like tensors."""
    g = generator(seed, device)
    for _ in range(count):
        u = torch.rand(shape, generator=g, device=device, dtype=torch.float32) - 0.5
        lap = -scale * torch.sign(u) * torch.log1p(-2.0 * u.abs())  # Laplace(0, scale) by inverse CDF
        z = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
        lap = torch.where(z < zero_frac, torch.zeros_like(lap), lap)
        s = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
        lap = torch.where(s < spike_frac, lap * spike, lap)
        yield lap.to(torch.bfloat16)


def bf16_bits(x: torch.Tensor):
    """Host numpy uint16 view of a BF16 tensor (for the oracle)."""
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
