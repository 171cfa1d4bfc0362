"""Bitwise-invariance checks and the difference metrics the pages' tracer
reports ("Batch-Invariant VLAs", section "Profiling batch-invariance": max and
mean absolute difference, RMSE, relative L2, output magnitude)."""
from __future__ import annotations

import torch


def row0_bit_equal(alone: torch.Tensor, batched_row0: torch.Tensor) -> bool:
    """True when two results have identical bits (NaN payloads included)."""
    if alone.shape != batched_row0.shape or alone.dtype != batched_row0.dtype:
        return False
    a = alone.contiguous().view(torch.uint8)
    b = batched_row0.contiguous().view(torch.uint8)
    return bool(torch.equal(a, b))


def diff_metrics(ref: torch.Tensor, other: torch.Tensor) -> dict:
    r = ref.double()
    o = other.double()
    d = (o - r).abs()
    rn = r.norm().item()
    return {
        "max_abs_diff": d.max().item() if d.numel() else 0.0,
        "mean_abs_diff": d.mean().item() if d.numel() else 0.0,
        "rmse": d.pow(2).mean().sqrt().item() if d.numel() else 0.0,
        "relative_l2": (d.norm().item() / rn) if rn else 0.0,
        "output_abs_max": r.abs().max().item() if r.numel() else 0.0,
    }
