"""Helpers shared by the parity tests: the error metrics and oracle calls on
sampled heads / time windows of large workloads.

Two metrics are computed for every comparison:
  * per slice: max over each (b, h) slice of max|x - ref| / max|ref| (the
    bar the tests assert: 1e-4 for fp32 inputs, 2e-2 for bf16 inputs);
  * element by element: max over elements of
    |x - ref| / max(|ref|, ELEM_FLOOR * max|ref of that slice|),
    which also sees rows far below their slice's maximum.
  * per row: max over rows (the last axis: a token-head's d values, or one
    state row) of max|x - ref| / max|ref| over the row, rows whose maximum is
    below ELEM_FLOOR of their slice's maximum left out (they are zero, or
    carry no information at the slice's scale).
All three are recorded per test and printed in the session summary
(conftest.py).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances of the parity bar: max relative error per (b, h) slice.
TOL_F32 = 1e-4
TOL_BF16 = 2e-2
# Floor of the element-by-element metric, relative to the slice maximum.
ELEM_FLOOR = 1e-3

# (test id, per-slice metric, element-by-element metric, per-row metric) of
# every comparison.
RECORDS: list[tuple[str, float, float, float]] = []
CURRENT = {"test": "?"}


def tol_for(dtype) -> float:
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact values of a (CPU or CUDA) tensor widened to fp64."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def _prep(x, ref, head_axes):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    other = tuple(i for i in range(x.ndim) if i not in head_axes)
    return x, ref, other


def elem_rel_err(x: np.ndarray, ref: np.ndarray, head_axes=(0, 2), floor: float = ELEM_FLOOR) -> float:
    """max over elements of |x - ref| / max(|ref|, floor * max|ref over the
    element's (b, h) slice|)."""
    x, ref, other = _prep(x, ref, head_axes)
    if not np.all(np.isfinite(x)):
        return float("inf")
    if x.size == 0:
        return 0.0
    smax = np.abs(ref).max(axis=other, keepdims=True)
    den = np.maximum(np.abs(ref), floor * smax)
    den = np.where(den > 0, den, 1.0)
    return float((np.abs(x - ref) / den).max())


def row_rel_err(x: np.ndarray, ref: np.ndarray, head_axes=(0, 2), floor: float = ELEM_FLOOR) -> float:
    """max over rows (last axis) of max|x - ref| / max|ref| within the row, for
    rows whose max|ref| is at least floor times their slice's maximum."""
    x, ref, other = _prep(x, ref, head_axes)
    if not np.all(np.isfinite(x)):
        return float("inf")
    if x.size == 0:
        return 0.0
    smax = np.abs(ref).max(axis=other, keepdims=True)
    rmax = np.abs(ref).max(axis=-1, keepdims=True)
    rerr = np.abs(x - ref).max(axis=-1, keepdims=True)
    keep = rmax >= floor * smax
    if not np.any(keep):
        return 0.0
    return float((rerr[keep] / np.where(rmax[keep] > 0, rmax[keep], 1.0)).max())


def max_rel_err(x: np.ndarray, ref: np.ndarray, head_axes=(0, 2)) -> float:
    """max over (b, h) slices of max|x - ref| / max|ref| (activations [B,T,H,d]).
    For states [B,H,d,d] pass head_axes=(0, 1).  Also records the
    element-by-element metric of the same pair for the session report."""
    x, ref, other = _prep(x, ref, head_axes)
    if not np.all(np.isfinite(x)):
        RECORDS.append((CURRENT["test"], float("inf"), float("inf"), float("inf")))
        return float("inf")
    if x.size == 0:
        return 0.0
    num = np.abs(x - ref).max(axis=other)
    den = np.abs(ref).max(axis=other)
    den = np.where(den > 0, den, 1.0)
    err = float((num / den).max())
    RECORDS.append((CURRENT["test"], err, elem_rel_err(x, ref, head_axes), row_rel_err(x, ref, head_axes)))
    return err


def gather_heads(t: torch.Tensor, pairs, t_lo: int, t_hi: int) -> np.ndarray:
    """[B,T,H,d] -> fp64 [1, t_hi - t_lo, n, d] holding the sampled (b, h) rows."""
    cols = [t[b, t_lo:t_hi, h, :] for (b, h) in pairs]
    return f64(torch.stack(cols, dim=1).unsqueeze(0))


def gather_state(s: torch.Tensor, pairs) -> np.ndarray:
    """[B,H,d,d] -> fp64 [1, n, d, d]."""
    return f64(torch.stack([s[b, h] for (b, h) in pairs], dim=0).unsqueeze(0))


def oracle_window(inp, gamma32, pairs, t_lo, t_hi, base, eps, state_in=None):
    """Oracle over tokens [t_lo, t_hi) of the sampled heads (positions preserved).
    Returns (y, o, state_out) shaped [1, W, n, d] / [1, n, d, d]."""
    g = np.array([float(gamma32[h]) for (_, h) in pairs], dtype=np.float64)
    args = [gather_heads(inp[n], pairs, t_lo, t_hi) for n in ("q", "k", "v", "gate")]
    return oracle.prefill(*args, g, state_in, pos_offset=t_lo, base=base, eps=eps)


def window_for(gamma32, pairs, rel: float = 1e-12) -> int:
    """Warm-up length W such that gamma^W <= rel for every sampled head: the
    state after W tokens from a zero start equals the true state up to rel."""
    gmax = max(float(gamma32[h]) for (_, h) in pairs)
    if gmax >= 1.0:
        raise ValueError("windowed comparison needs gamma < 1")
    return int(np.ceil(np.log(rel) / np.log(gmax)))
