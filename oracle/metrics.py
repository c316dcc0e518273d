"""Parity metrics.

TEST INFRASTRUCTURE ONLY (see the package header).

  max relative error = max|g - r| / max|r|
  relative L2        = ||g - r||_2 / ||r||_2
  PSNR               = 20 log10(peak / RMSE), peak = max(r) - min(r) of the reference (random
                       weights give no [-1, 1] range to take the peak from)
"""
from __future__ import annotations

import numpy as np


def max_rel(g: np.ndarray, r: np.ndarray) -> float:
    r = np.asarray(r, dtype=np.float64)
    d = np.abs(np.asarray(g, dtype=np.float64) - r).max() if r.size else 0.0
    m = np.abs(r).max() if r.size else 0.0
    return float(d / m) if m > 0 else float(d)


def rel_l2(g: np.ndarray, r: np.ndarray) -> float:
    r = np.asarray(r, dtype=np.float64)
    d = np.asarray(g, dtype=np.float64) - r
    n = np.sqrt((r * r).sum())
    return float(np.sqrt((d * d).sum()) / n) if n > 0 else float(np.sqrt((d * d).sum()))


def psnr(g: np.ndarray, r: np.ndarray) -> float:
    r = np.asarray(r, dtype=np.float64)
    d = np.asarray(g, dtype=np.float64) - r
    rmse = np.sqrt((d * d).mean())
    peak = r.max() - r.min()
    if rmse == 0:
        return float("inf")
    return float(20.0 * np.log10(peak / rmse))
