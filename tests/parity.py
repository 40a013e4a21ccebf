"""Comparison rule between the CUDA path's y and the oracle's y.

The contract lets the FP32 summation order vary ("Tensor Programs, Part 1",
rule 1), so several y are correct.  Rule used here:
  * bit-exact (up to +0 == -0) when every FP32 partial sum is exact, e.g.
    small-integer inputs;
  * otherwise |y - y_ref| <= 2 * ulp16(max(|p_ref|, |y_ref|)), where p_ref is
    the oracle's rounded projection and ulp16(v) is the binary16 spacing at
    |v| (2^-24 below 2^-14).  Using the larger of |p| and |y| covers
    cancellation in y = p + b, where one ulp of p lands in y unchanged.
  * infinities must match exactly; NaN must meet NaN.
"""
from __future__ import annotations

import numpy as np


def ulp16(v: np.ndarray) -> np.ndarray:
    a = np.abs(v.astype(np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -14.0)
    return np.exp2(e - 10.0)


def compare(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, p_ref_bits: np.ndarray | None,
            exact: bool, max_ulps: float = 2.0):
    """Returns (ok, report) for binary16 bit arrays of equal shape."""
    g = y_gpu_bits.view(np.float16).astype(np.float64)
    r = y_ref_bits.view(np.float16).astype(np.float64)
    nan_g, nan_r = np.isnan(g), np.isnan(r)
    bad = nan_g != nan_r
    fin = ~(nan_g | nan_r)
    inf_mismatch = fin & (np.isinf(g) | np.isinf(r)) & (g != r)
    bad |= inf_mismatch
    both = fin & ~np.isinf(g) & ~np.isinf(r)
    diff = np.zeros_like(g)
    diff[both] = np.abs(g[both] - r[both])
    if exact:
        bad |= both & (diff != 0)
        tol_ulps = np.zeros_like(g)
    else:
        mag = np.abs(r)
        if p_ref_bits is not None:
            p = p_ref_bits.view(np.float16).astype(np.float64)
            p = np.where(np.isfinite(p), np.abs(p), 0.0)
            mag = np.maximum(mag, p)
        u = ulp16(mag)
        bad |= both & (diff > max_ulps * u)
        tol_ulps = np.where(both, diff / u, 0.0)
    n_bad = int(bad.sum())
    report = {
        "elements": int(g.size),
        "bad": n_bad,
        "exact_match": int((both & (diff == 0)).sum()),
        "max_ulps": float(tol_ulps.max()) if g.size else 0.0,
    }
    if n_bad:
        idx = np.argwhere(bad)[:5]
        report["first_bad"] = [(tuple(int(i) for i in ix), float(g[tuple(ix)]), float(r[tuple(ix)]))
                               for ix in idx]
    return n_bad == 0, report
