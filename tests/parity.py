"""Comparison rule between the CUDA path's y and the oracle's y.

The contract lets the FP32 summation order vary ("Tensor Programs, Part 1",
rule 1), so several y are correct.  Rule used here:
  * bit-exact (up to +0 == -0) when every FP32 partial sum is exact, e.g.
    small-integer inputs;
  * otherwise |y - y_ref| <= 2 * ulp16(max(|p_ref|, |y_ref|)), where p_ref is
    the oracle's rounded projection and ulp16(v) is the binary16 spacing at
    |v| (2^-24 below 2^-14).  Using the larger of |p| and |y| covers
    cancellation in y = p + b, where one ulp of p lands in y unchanged.
  * an element beyond 2 ulps passes only if it lies inside the interval that
    holds every result of an FP32 accumulation of the same products
    (``legal_interval``), and such elements must stay rare (``max_outside``).
    They arise where the sum cancels (|S| much smaller than sum |x w|) and the
    tensor core's FP32 accumulation, whose alignment of addends truncates,
    differs from the oracle's sequential round-to-nearest sum.
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


def legal_interval(x16: np.ndarray, w16: np.ndarray, b16: np.ndarray):
    """[lo, hi] per element holding y for any FP32 accumulation of the products.

    S and A = sum |x w| in binary64 (products of binary16 numbers are exact;
    the binary64 sum errs by at most K 2^-53 A, covered by a margin).  An
    FP32 accumulation of K products with unit roundoff u errs by at most
    gamma_K A, gamma_K = K u / (1 - K u) (Higham, "Accuracy and Stability of
    Numerical Algorithms", section 3.1).  u = 2^-23 also covers accumulators
    that truncate instead of rounding.  RN16 is monotone, so
    y lies in [RN16(RN16(S - E) + b), RN16(RN16(S + E) + b)].
    """
    x = x16.astype(np.float64)
    w = w16.astype(np.float64)
    K = x.shape[1]
    S = x @ w.T
    A = np.abs(x) @ np.abs(w).T
    u = 2.0 ** -23
    gamma = K * u / (1 - K * u)
    E = gamma * A + A * 2.0 ** -40
    bb = b16.astype(np.float64)[None, :]
    with np.errstate(over="ignore", invalid="ignore"):
        lo = ((S - E).astype(np.float16).astype(np.float64) + bb).astype(np.float16).astype(np.float64)
        hi = ((S + E).astype(np.float16).astype(np.float64) + bb).astype(np.float16).astype(np.float64)
    return lo, hi


def compare(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, p_ref_bits: np.ndarray | None,
            exact: bool, max_ulps: float = 2.0, interval=None, max_outside: float = 1e-4):
    """Returns (ok, report) for binary16 bit arrays of equal shape.

    interval: optional (lo, hi) from ``legal_interval``; elements beyond
    ``max_ulps`` then pass if inside it, as long as their fraction stays at
    or below ``max_outside``.
    """
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
        beyond = both & (diff > max_ulps * u)
        n_beyond = int(beyond.sum())
        n_inside = 0
        if interval is not None:
            lo, hi = interval
            inside = (g >= lo) & (g <= hi)
            n_inside = int((beyond & inside).sum())
            bad |= beyond & ~inside
            if n_beyond > max_outside * max(1, g.size):
                bad |= beyond
        else:
            bad |= beyond
        tol_ulps = np.where(both, diff / u, 0.0)
    n_bad = int(bad.sum())
    report = {
        "elements": int(g.size),
        "bad": n_bad,
        "exact_match": int((both & (diff == 0)).sum()),
        "max_ulps": float(tol_ulps.max()) if g.size else 0.0,
    }
    if not exact:
        report["beyond_2ulp"] = n_beyond
        report["beyond_2ulp_inside_interval"] = n_inside
    if n_bad:
        idx = np.argwhere(bad)[:5]
        report["first_bad"] = [(tuple(int(i) for i in ix), float(g[tuple(ix)]), float(r[tuple(ix)]))
                               for ix in idx]
    return n_bad == 0, report
