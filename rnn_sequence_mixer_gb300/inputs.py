"""Seeded synthetic inputs shared by the CUDA path and the oracle.

This module holds none of the mixer's arithmetic: it only draws N(0, 1)
tensors from a seeded ``torch.Generator`` and rounds them to the workload's
dtype (round-to-nearest-even for bf16).  The tests hand the exact same bits to
the library and, widened to fp64, to the oracle.
"""
from __future__ import annotations

import torch


def normal(shape, dtype, gen: torch.Generator, device) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return x.to(dtype)


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def mixer_inputs(B, T, H, d, dtype, seed, device="cpu", with_dy=False):
    """q, k, v, gate (and dy) of shape [B, T, H, d], drawn in that order."""
    gen = generator(seed, device)
    names = ["q", "k", "v", "gate"] + (["dy"] if with_dy else [])
    return {n: normal((B, T, H, d), dtype, gen, device) for n in names}


def state(B, H, d, seed, scale=1.0, device="cpu") -> torch.Tensor:
    """A seeded fp32 [B, H, d, d] state (for tests that start from a non-zero state)."""
    gen = generator(seed, device)
    return normal((B, H, d, d), torch.float32, gen, device) * scale


def decode_inputs(steps, B, H, d, dtype, seed, device="cpu"):
    """Per-step decode rows: q, k, v, gate of shape [steps, B, 1, H, d] (each
    step's slice is contiguous), drawn in that order."""
    gen = generator(seed, device)
    return {n: normal((steps, B, 1, H, d), dtype, gen, device) for n in ("q", "k", "v", "gate")}
