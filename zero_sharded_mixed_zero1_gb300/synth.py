"""Seeded synthetic inputs for the optimizer step.

This module only draws random numbers; it holds none of the step's arithmetic.
bf16 gradients are made by truncating fp32 normal draws to their upper 16
bits (a distribution choice, not the step's round-to-nearest-even).  Draws use
torch generators on the target device, so the same seed gives the same tensor
on every call on that device type.
"""
from __future__ import annotations

import numpy as np
import torch


def seed_of(*keys: int) -> int:
    """A 63-bit seed derived from a tuple of non-negative integers."""
    return int(np.random.SeedSequence([int(k) for k in keys]).generate_state(2, np.uint64)[0] >> np.uint64(1))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_f32(n: int, std: float, seed: int, device="cpu") -> torch.Tensor:
    """n fp32 draws from N(0, std^2)."""
    x = torch.randn(n, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return x.mul_(std)


def truncate_to_bf16(x: torch.Tensor) -> torch.Tensor:
    """The upper 16 bits of each fp32 value, as bfloat16."""
    return (x.contiguous().view(torch.int32) >> 16).to(torch.int16).view(torch.bfloat16)


def normal_bf16(n: int, std: float, seed: int, device="cpu") -> torch.Tensor:
    """n bf16 values: N(0, std^2) draws truncated to bf16."""
    return truncate_to_bf16(normal_f32(n, std, seed, device))


def set_inf(x: torch.Tensor, p: float, seed: int) -> int:
    """Set each element of a bf16 tensor to +inf with probability p (in
    place); returns how many were set."""
    mask = torch.rand(x.numel(), generator=_gen(seed, x.device), device=x.device) < p
    x.view(-1)[mask] = float("inf")
    return int(mask.sum())
