"""Seeded synthetic inputs for the qpack workloads.

This module only draws random tensors (weights and activations) with the distributions and shapes of the
workloads; it holds none of the quantization arithmetic. Tests hand the same tensors to the CUDA path and to
the CPU oracle, so the two never need bit-identical random streams: the oracle always receives a byte copy.

Distributions:
- normal(std): torch's Gaussian sampler.
- laplace(b): inverse CDF of a uniform draw, x = -b * sign(u) * log(1 - 2|u|), u ~ U(-1/2, 1/2).
- outlier matrix: N(0, std^2) with exactly floor(frac * numel) distinct positions replaced by
  ±U(lo, hi) with a random sign.
"""
from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def laplace(shape, b: float, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    g = _gen(seed, device)
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float32) - 0.5
    # keep |u| < 1/2 so the log stays finite
    u = u.clamp_(-0.49999997, 0.49999997)
    x = -b * torch.sign(u) * torch.log1p(-2.0 * u.abs())
    return x.to(dtype)


def normal_with_outliers(shape, std: float, frac: float, lo: float, hi: float, seed: int,
                         device="cpu") -> torch.Tensor:
    """N(0, std^2) fp32 with floor(frac * numel) distinct entries replaced by ±U(lo, hi)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    n = 1
    for s in shape:
        n *= int(s)
    w = torch.randn(n, generator=g, dtype=torch.float32) * std
    n_out = int(frac * n)
    pos = torch.randperm(n, generator=g)[:n_out]
    mag = lo + (hi - lo) * torch.rand(n_out, generator=g, dtype=torch.float32)
    sign = torch.where(torch.rand(n_out, generator=g) < 0.5, -1.0, 1.0)
    w[pos] = sign * mag
    return w.reshape(shape).to(device)


def seed_for(*parts: int) -> int:
    """Combine small integers (config id, layer id, matrix index) into one 63-bit seed."""
    s = 0x5151_AC4B
    for p in parts:
        s = (s * 1_000_003 + int(p) + 1) % (1 << 63)
    return s
