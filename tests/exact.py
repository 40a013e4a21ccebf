"""Exact rational arithmetic and fixture parsing used by the tests.

Everything here is written independently of ``oracle/`` and of the CUDA
path: binary16 decoding from the bit fields, rounding of an exact rational
to binary16 by the IEEE 754 definition, and the error interval of a
recursively summed binary32 dot product (Higham, "Accuracy and Stability of
Numerical Algorithms", 2nd ed., section 3.1: |fl(S) - S| <= gamma_n sum|x_k w_k|
with gamma_n = n u / (1 - n u), u = 2^-24).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F16_MAX = Fraction(65504)
U32 = Fraction(1, 2 ** 24)


def f16_bits_to_fraction(h: int):
    """Exact value of a finite binary16 bit pattern (None for inf/NaN)."""
    h = int(h) & 0xFFFF
    s = -1 if h >> 15 else 1
    e = (h >> 10) & 0x1F
    f = h & 0x3FF
    if e == 31:
        return None
    if e == 0:
        return s * Fraction(f, 2 ** 24)
    return s * Fraction(1024 + f, 2 ** 10) * Fraction(2) ** (e - 15)


def rn16(q: Fraction) -> float:
    """Round an exact rational to binary16, nearest, ties to even.

    Returns a Python float (every binary16 value is exact in a double);
    +-inf on overflow; +0.0 for zero (the sign of an exact zero is the
    caller's business).
    """
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(q)
    p = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** p > a:
        p -= 1
    while Fraction(2) ** (p + 1) <= a:
        p += 1
    qexp = -24 if p < -14 else p - 10
    n = a / Fraction(2) ** qexp
    whole = n.numerator // n.denominator
    rem = n - whole
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and whole % 2 == 1):
        whole += 1
    val = Fraction(whole) * Fraction(2) ** qexp
    if val > F16_MAX:
        return sign * math.inf
    return sign * float(val)


def exact_sums(x_bits: np.ndarray, w_bits: np.ndarray):
    """S[m][n] = sum_k x[m,k] w[n,k] exactly, and A[m][n] = sum_k |x w|."""
    M, K = x_bits.shape
    N = w_bits.shape[0]
    xf = [[f16_bits_to_fraction(v) for v in row] for row in x_bits]
    wf = [[f16_bits_to_fraction(v) for v in row] for row in w_bits]
    S = [[sum((xf[m][k] * wf[n][k] for k in range(K)), Fraction(0)) for n in range(N)]
         for m in range(M)]
    A = [[sum((abs(xf[m][k] * wf[n][k]) for k in range(K)), Fraction(0)) for n in range(N)]
         for m in range(M)]
    return S, A


def exact_linear(x_bits, w_bits, b_bits):
    """y = RN16(RN16(S) + b) with S exact: the contract when no sum rounds."""
    S, _ = exact_sums(x_bits, w_bits)
    M, N = len(S), len(S[0]) if S else 0
    y = np.zeros((M, N), dtype=np.float64)
    for m in range(M):
        for n in range(N):
            p = rn16(S[m][n])
            bv = f16_bits_to_fraction(b_bits[n])
            if math.isinf(p):
                y[m, n] = p
            else:
                y[m, n] = rn16(Fraction(p) + bv)
    return y


def higham_interval(x_bits, w_bits, b_bits):
    """Per element [lo, hi] holding every legal y for any FP32 summation order.

    With E = gamma_K * sum|x w|, the computed FP32 sum lies in [S-E, S+E];
    RN16 is monotone, so y lies between RN16(RN16(S-E)+b) and RN16(RN16(S+E)+b).
    """
    K = x_bits.shape[1]
    S, A = exact_sums(x_bits, w_bits)
    gamma = (K * U32) / (1 - K * U32)
    M, N = len(S), len(S[0]) if S else 0
    lo = np.zeros((M, N))
    hi = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            E = gamma * A[m][n]
            bv = f16_bits_to_fraction(b_bits[n])
            for dst, v in ((lo, S[m][n] - E), (hi, S[m][n] + E)):
                p = rn16(v)
                dst[m, n] = p if math.isinf(p) else rn16(Fraction(p) + bv)
    return lo, hi


def parse_golden(name: str):
    """Read a tests/golden fixture: returns (x, w, b, y) as float16 / float64."""
    path = os.path.join(GOLDEN_DIR, name)
    sections: dict[str, list[list[float]]] = {}
    dims: dict[str, int] = {}
    cur = None
    with open(path) as fh:
        for raw in fh:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] in ("M", "N", "K") and len(tok) == 2:
                dims[tok[0]] = int(tok[1])
                continue
            if tok[0] in ("x", "w", "b", "y") and len(tok) == 1:
                cur = tok[0]
                sections[cur] = []
                continue
            sections[cur].append([float(t) for t in tok])
    M, N, K = dims["M"], dims["N"], dims["K"]
    x = np.array(sections["x"], dtype=np.float64).reshape(M, K)
    w = np.array(sections["w"], dtype=np.float64).reshape(N, K)
    b = np.array(sections["b"], dtype=np.float64).reshape(N)
    y = np.array(sections["y"], dtype=np.float64).reshape(M, N)
    for arr in (x, w, b, y):
        # fixtures hold exact binary16 values only
        finite = np.isfinite(arr)
        assert np.array_equal(arr[finite].astype(np.float16).astype(np.float64), arr[finite]), name
    return x.astype(np.float16), w.astype(np.float16), b.astype(np.float16), y


def same_values(a, b) -> bool:
    """Element-wise equality of binary16 results, +0 == -0, NaN == NaN."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return bool(np.all((a == b) | (np.isnan(a) & np.isnan(b))))


# ---- formats other than binary16 -------------------------------------------------
# (p significand bits with the hidden bit, minimum normal exponent, maximum exponent)
FORMATS = {"f16": (11, -14, 15), "bf16": (8, -126, 127)}


def rn_format(q, fmt: str) -> float:
    """Round an exact rational (or float) to binary16 / bfloat16, nearest even.

    Returns a Python float (exact for both formats); +-inf on overflow.
    """
    p, emin, emax = FORMATS[fmt]
    q = Fraction(q)
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    qe = max(e, emin) - (p - 1)
    n = a / Fraction(2) ** qe
    whole = n.numerator // n.denominator
    rem = n - whole
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and whole % 2 == 1):
        whole += 1
    val = Fraction(whole) * Fraction(2) ** qe
    maxv = (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    if val > maxv:
        return sign * math.inf
    return sign * float(val)


def bf16_bits_to_float(h) -> np.ndarray:
    """bfloat16 bit patterns -> float64 values (bfloat16 is binary32's upper half)."""
    h = np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16
    return h.view(np.float32).astype(np.float64)


def float_to_bits(v, fmt: str) -> np.ndarray:
    """Exact binary16 / bfloat16 values (float64) -> their bit patterns."""
    v = np.asarray(v, dtype=np.float64)
    if fmt == "f16":
        return v.astype(np.float16).view(np.uint16)
    f = v.astype(np.float32)
    assert np.array_equal(f.astype(np.float64)[np.isfinite(v)], v[np.isfinite(v)])
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def parse_chain_golden(name: str):
    """Read 'case <dtype> <op> <t> <y>' lines of an epilogue fixture."""
    cases = []
    with open(os.path.join(GOLDEN_DIR, name)) as fh:
        for raw in fh:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            assert tok[0] == "case" and len(tok) == 5, line
            cases.append((tok[1], tok[2], float(tok[3]), float(tok[4])))
    return cases
