"""Comparison rule between the CUDA path's y and the oracle's y -- TEST
INFRASTRUCTURE ONLY (used by ``tests/`` and by the parity leg of
``bench.py``, like the rest of this package).

The contract lets the FP32 summation order vary ("Tensor Programs, Part 1",
section "One Program and One Numerical Contract", rule 1), so several y are
correct.  The rule:
  * bit-exact (up to +0 == -0) when every FP32 partial sum is exact, e.g.
    small-integer inputs;
  * otherwise |y - y_ref| <= 2 * ulp16(max(|p_ref|, |y_ref|)), where p_ref is
    the oracle's rounded projection and ulp16(v) is the binary16 spacing at
    |v| (2^-24 below 2^-14).  Using the larger of |p| and |y| covers
    cancellation in y = p + b, where one ulp of p lands in y unchanged.
  * an element beyond 2 ulps passes only if it lies inside the interval that
    holds every result of an IEEE round-to-nearest FP32 accumulation of the
    same products in any order (``legal_interval``, unit roundoff
    u = 2^-24), and such elements must stay rare (``max_outside``).  They
    arise where the sum cancels (|S| much smaller than sum |x w|): two legal
    FP32 orders already differ by more than 2 FP16 ulps there.
  * infinities must match exactly; NaN must meet NaN.

Besides pass / fail, a report counts the elements beyond 2 ulps of y_ref
alone (the literal reading of "within 2 FP16 ULP of the oracle's y") with
the largest such difference; where y = p + b cancels these are large in
ulps of y and small in ulps of p.  ``intervals`` also gives the wider
interval with u = 2^-23, which bounds an accumulator that truncates instead
of rounding; it is a diagnostic and decides nothing.
"""
from __future__ import annotations

import numpy as np

U_RN = 2.0 ** -24     # unit roundoff of binary32 round-to-nearest
U_TRUNC = 2.0 ** -23  # one binary32 ulp: bounds an accumulator that truncates


def ulp16(v: np.ndarray) -> np.ndarray:
    a = np.abs(v.astype(np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -14.0)
    return np.exp2(e - 10.0)


def _f64(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.float16)
    return a.astype(np.float64)


def _sums(x16: np.ndarray, w16: np.ndarray):
    x, w = _f64(x16), _f64(w16)
    return x @ w.T, np.abs(x) @ np.abs(w).T, x.shape[1]


def _interval_from(S, A, K, b16, u):
    gamma = K * u / (1 - K * u)
    E = gamma * A + A * 2.0 ** -40
    bb = _f64(b16)[None, :]
    with np.errstate(over="ignore", invalid="ignore"):
        lo = ((S - E).astype(np.float16).astype(np.float64) + bb).astype(np.float16).astype(np.float64)
        hi = ((S + E).astype(np.float16).astype(np.float64) + bb).astype(np.float16).astype(np.float64)
    return lo, hi


def legal_interval(x16: np.ndarray, w16: np.ndarray, b16: np.ndarray, u: float = U_RN):
    """[lo, hi] per element holding y for any FP32 accumulation of the products.

    S and A = sum |x w| in binary64 (products of binary16 numbers are exact;
    the binary64 sum errs by at most K 2^-53 A, covered by a margin).  An
    FP32 accumulation of K products with unit roundoff u errs by at most
    gamma_K A, gamma_K = K u / (1 - K u) (Higham, "Accuracy and Stability of
    Numerical Algorithms", section 3.1).  The default u = 2^-24 is binary32
    round-to-nearest; u = 2^-23 would also cover an accumulator that
    truncates.  RN16 is monotone, so y lies in
    [RN16(RN16(S - E) + b), RN16(RN16(S + E) + b)].
    """
    S, A, K = _sums(x16, w16)
    return _interval_from(S, A, K, b16, u)


def intervals(x16: np.ndarray, w16: np.ndarray, b16: np.ndarray):
    """(interval with u = 2^-24, the rule's; interval with u = 2^-23, the
    truncating accumulator's, a diagnostic), sums computed once."""
    S, A, K = _sums(x16, w16)
    return _interval_from(S, A, K, b16, U_RN), _interval_from(S, A, K, b16, U_TRUNC)


def compare(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, p_ref_bits: np.ndarray | None,
            exact: bool, max_ulps: float = 2.0, interval=None, max_outside: float = 1e-4,
            wide_interval=None):
    """Returns (ok, report) for binary16 bit arrays of equal shape.

    interval: optional (lo, hi) from ``legal_interval``; elements beyond
    ``max_ulps`` then pass if inside it, as long as their fraction stays at
    or below ``max_outside``.  wide_interval: optional (lo, hi) with
    u = 2^-23; only counted (``beyond_2ulp_outside_truncating_interval``).
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
    n_beyond = n_inside = 0
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
    # the literal reading: differences in ulps of y_ref alone
    y_ulps = np.where(both, diff / ulp16(r), 0.0)
    report = {
        "elements": int(g.size),
        "bad": n_bad,
        "exact_match": int((both & (diff == 0)).sum()),
        "max_ulps": float(tol_ulps.max()) if g.size else 0.0,
        "beyond_2ulp_of_y": int((y_ulps > max_ulps).sum()),
        "max_ulps_of_y": float(y_ulps.max()) if g.size else 0.0,
    }
    if not exact:
        report["beyond_2ulp"] = n_beyond
        report["beyond_2ulp_inside_interval"] = n_inside
        if interval is not None:
            report["beyond_2ulp_outside_interval"] = n_beyond - n_inside
        if wide_interval is not None:
            lo, hi = wide_interval
            report["beyond_2ulp_outside_truncating_interval"] = int((beyond & ((g < lo) | (g > hi))).sum())
    if n_bad:
        idx = np.argwhere(bad)[:5]
        report["first_bad"] = [(tuple(int(i) for i in ix), float(g[tuple(ix)]), float(r[tuple(ix)]))
                               for ix in idx]
    return n_bad == 0, report


def judge(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, p_ref_bits: np.ndarray, x16: np.ndarray,
          w16: np.ndarray, b16: np.ndarray, exact: bool, max_outside: float = 1e-5):
    """``compare`` for oracle results already at hand (x16: the rows they cover).

    The legal interval is computed only for rows that hold an element
    beyond 2 ulps, so large row samples stay cheap.  Returns (ok, report).
    """
    if exact:
        return compare(y_gpu_bits, y_ref_bits, p_ref_bits, exact=True)
    ok0, rep0 = compare(y_gpu_bits, y_ref_bits, p_ref_bits, exact=False, max_outside=max_outside)
    if ok0:
        rep0["beyond_2ulp_outside_interval"] = 0
        return ok0, rep0
    g = y_gpu_bits.view(np.float16).astype(np.float64)
    r = y_ref_bits.view(np.float16).astype(np.float64)
    p = p_ref_bits.view(np.float16).astype(np.float64)
    mag = np.maximum(np.abs(r), np.abs(np.where(np.isfinite(p), p, 0.0)))
    with np.errstate(invalid="ignore"):
        flagged = ~(np.abs(g - r) <= 2 * ulp16(mag))
    rsel = np.unique(np.nonzero(flagged)[0])
    iv_rn, iv_t = intervals(np.asarray(x16)[rsel], w16, b16)
    full_rn = (np.full(g.shape, -np.inf), np.full(g.shape, np.inf))
    full_t = (np.full(g.shape, -np.inf), np.full(g.shape, np.inf))
    full_rn[0][rsel], full_rn[1][rsel] = iv_rn
    full_t[0][rsel], full_t[1][rsel] = iv_t
    return compare(y_gpu_bits, y_ref_bits, p_ref_bits, exact=False, interval=full_rn, max_outside=max_outside,
                   wide_interval=full_t)


def check_rows(y_gpu_bits: np.ndarray, x16: np.ndarray, w16: np.ndarray, b16: np.ndarray, exact: bool,
               rows=None, max_outside: float = 1e-5, nthreads: int | None = None):
    """Oracle on ``rows`` of x (all rows when None), then ``judge``.

    y_gpu_bits holds the CUDA path's y for exactly those rows.
    Returns (ok, report).
    """
    from . import linear_f16  # the oracle itself

    x = np.asarray(x16)
    if rows is not None:
        x = x[np.asarray(rows)]
    x = np.ascontiguousarray(x)
    yr, pr = linear_f16(x, w16, b16, want_proj=True, nthreads=nthreads)
    return judge(y_gpu_bits, yr, pr, x, w16, b16, exact, max_outside)
