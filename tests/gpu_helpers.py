"""Helpers shared by the GPU parity tests: the tolerance the results are held
to, and small utilities.  The expected values always come from the fp64 CPU
oracle (``oracle``), never from the CUDA path.

Tolerance (per element, from the fp64 oracle value ``ref`` and
``absum = |alpha| * sum_k |a_k b_k| (+ |bias|)``):
    fp32 output:  |c - ref| <= 1e-4 * absum
    bf16 output:  |c - ref| <= 1e-4 * absum + 2^-8 * |ref|
    fp16 output:  |c - ref| <= 1e-4 * absum + 2^-11 * |ref| + 2^-25
The 1e-4 * absum term covers fp32 accumulation over up to 8192 terms (worst
case K/16 accumulator roundings of at most 2^-23 relative each: 512 * 1.2e-7
= 6.1e-5 < 1e-4); 2^-8 |ref| is half a bf16 unit in the last place, the final
rounding; for fp16 output 2^-11 |ref| is half an fp16 unit in the last place
and 2^-25 half its subnormal spacing.
"""
from __future__ import annotations

import numpy as np
import torch


def check_tolerance(gpu: torch.Tensor, ref: np.ndarray, absum: np.ndarray, what: str = "") -> float:
    """Asserts the tolerance; returns the worst normalised error (error / bound)."""
    g = gpu.detach().to("cpu", torch.float64).numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    bound = 1e-4 * absum
    if gpu.dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * np.abs(ref)
    elif gpu.dtype == torch.float16:
        bound = bound + 2.0 ** -11 * np.abs(ref) + 2.0 ** -25
    err = np.abs(g - ref)
    bad = ~(err <= bound)  # NaN counts as a failure
    if bad.any():
        idx = np.argwhere(bad)[:5]
        details = [(tuple(i), g[tuple(i)], ref[tuple(i)], bound[tuple(i)]) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, e.g. {details}")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, 0.0)
    return float(ratio.max()) if ratio.size else 0.0


def bits_equal(x: torch.Tensor, y: torch.Tensor) -> bool:
    if x.shape != y.shape or x.dtype != y.dtype:
        return False
    return bool(torch.equal(x.contiguous().view(torch.uint8), y.contiguous().view(torch.uint8)))


def padded(rows: int, cols: int, pad_cols: int, dtype=torch.bfloat16, device="cuda", fill=0.0):
    """A [rows, cols] view into [rows, pad_cols] storage (row stride pad_cols)."""
    store = torch.full((rows, pad_cols), fill, dtype=dtype, device=device)
    return store, store[:, :cols]
