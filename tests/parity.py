"""Shared helpers of the parity tests: tolerances and comparison against the oracle.

Tolerances (fp32 accumulation in every kernel):
  fp32:  |y - ref| <= 1e-5 * A + 1e-6
  fp16:  |y - ref| <= 2e-3 * |ref| + 1e-3 * A / sqrt(Kg)
where ref is the oracle's unrounded fp64 result, A = sum |x * w| over the taps of that
output and Kg = (C / group) * prod(kernel) the per-group reduction length.
ThresholdedRelu is discontinuous at alpha: where |v_ref - alpha| is within the
tolerance either branch is accepted.
"""
from __future__ import annotations

import math

import numpy as np


def tolerance(ref: np.ndarray, absacc: np.ndarray, dtype: str, kg: int) -> np.ndarray:
    if dtype == "f32":
        return 1e-5 * absacc + 1e-6
    return 2e-3 * np.abs(ref) + 1e-3 * absacc / math.sqrt(kg)


def check(y: np.ndarray, ref: np.ndarray, absacc: np.ndarray, dtype: str, kg: int,
          activation=None, alpha: float = 1.0, pre_act: np.ndarray | None = None,
          what: str = "") -> None:
    """Assert y matches ref element by element within the stated tolerance."""
    y = np.asarray(y, dtype=np.float64)
    assert y.shape == ref.shape, (what, y.shape, ref.shape)
    tol = tolerance(ref, absacc, dtype, kg)
    err = np.abs(y - ref)
    bad = ~(err <= tol)
    if activation == "ThresholdedRelu" and pre_act is not None:
        # either side of the jump is correct when v is within tolerance of alpha
        near = np.abs(pre_act - alpha) <= tolerance(pre_act, absacc, dtype, kg)
        ok_other = np.abs(y - np.where(ref == 0.0, pre_act, 0.0)) <= tol
        bad &= ~(near & ok_other)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        lines = [f"{tuple(i)}: y={y[tuple(i)]!r} ref={ref[tuple(i)]!r} tol={tol[tuple(i)]!r}"
                 for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs out of "
                             f"tolerance (max err {float(err.max()):.3e})\n" + "\n".join(lines))
