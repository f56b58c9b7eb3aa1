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


def layer_inputs(B, T, D, H, d, seed, device="cpu", with_dy=False):
    """Inputs of one RNN layer with its projections: x [B, T, D], the input
    weights w_qkvz [H, 4, d, D] and the output weight w_o [D, H d], all bf16,
    drawn in that order (and dy [B, T, H, d]).  The weights are N(0, 1) / sqrt
    of their fan-in, so the projected rows are about N(0, 1)."""
    gen = generator(seed, device)
    out = {"x": normal((B, T, D), torch.bfloat16, gen, device),
           "w_qkvz": (torch.randn((H, 4, d, D), generator=gen, device=device) / D ** 0.5).to(torch.bfloat16),
           "w_o": (torch.randn((D, H * d), generator=gen, device=device) / (H * d) ** 0.5).to(torch.bfloat16)}
    if with_dy:
        out["dy"] = normal((B, T, H, d), torch.bfloat16, gen, device)
    return out
