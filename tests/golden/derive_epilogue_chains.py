#!/usr/bin/env python
"""Derivation of the golden epilogue chains (epilogue_silu.txt,
epilogue_gelu.txt): every primitive of SiLU and GELU evaluated exactly in
rationals and rounded to the head dtype, as the ContractionEpilogue row of
the OpKind table reads ("ML compiler internals", section "The OpKind
vocabulary": the head keeps its dtype and every step rounds through it) and
section "SwiGLU and GeLU FFN" builds the activations from primitives.

Independent of the oracle and of the CUDA package: Python's fractions for
the arithmetic, and math.exp / math.erf (binary64, within an ulp of the true
value) for the two transcendental primitives; every case prints the
position of its value between two representable neighbours, so a reader can
see that no rounding decision lies near a tie.

    python tests/golden/derive_epilogue_chains.py

prints each derivation as the fixtures' comment lines and then the fixtures'
"case" lines, which tests/test_oracle_contraction.py compares with the
committed files.
"""
from __future__ import annotations

import math
from fractions import Fraction as Q

# significand bits (with the hidden one) and the smallest normal exponent
FORMATS = {"f16": (11, -14), "bf16": (8, -126)}


def round_even(q: Q, dtype: str):
    """q rounded to the nearest value of the format, ties to even
    (overflow does not arise in these cases).  Returns (value, note)."""
    p, emin = FORMATS[dtype]
    if q == 0:
        return Q(0), "exact"
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Q(2) ** e > a:
        e -= 1
    while Q(2) ** (e + 1) <= a:
        e += 1
    quantum_exp = max(e, emin) - (p - 1)
    n = a / Q(2) ** quantum_exp          # the value in quanta
    whole = n.numerator // n.denominator
    frac = n - whole
    if frac > Q(1, 2) or (frac == Q(1, 2) and whole % 2 == 1):
        whole += 1
    value = sign * whole * Q(2) ** quantum_exp
    if frac == 0:
        return value, "exact"
    return value, f"quantum 2^{quantum_exp}, {float(n):.3f} -> {whole}"


class Chain:
    def __init__(self, dtype: str):
        self.dtype = dtype
        self.lines = []

    def step(self, name: str, exact: Q, text: str) -> Q:
        v, note = round_even(exact, self.dtype)
        self.lines.append(f"#   {name} = RN({text} = {float(exact):.10g}): {note} -> {float(v)!r}")
        return v


def exp_q(v: Q) -> Q:
    return Q(math.exp(float(v)))


def erf_q(v: Q) -> Q:
    return Q(math.erf(float(v)))


def silu(t: Q, dtype: str):
    c = Chain(dtype)
    a = c.step("a", -t, "-t")
    e = c.step("e", exp_q(a), "exp(a)")
    d = c.step("d", 1 + e, "1 + e")
    return c.step("y", t / d, "t / d"), c.lines


def gelu_tanh(t: Q, dtype: str):
    c = Chain(dtype)
    c1 = c.step("c1", Q(0.044715), "0.044715")
    c2 = c.step("c2", Q(2 * math.sqrt(2 / math.pi)), "2 sqrt(2/pi)")
    s = c.step("s", t * t, "t * t")
    cu = c.step("c", s * t, "s * t")
    u = c.step("u", c1 * cu, "c1 * c")
    v = c.step("v", t + u, "t + u")
    z = c.step("z", c2 * v, "c2 * v")
    a = c.step("a", -z, "-z")
    e = c.step("e", exp_q(a), "exp(a)")
    d = c.step("d", 1 + e, "1 + e")
    return c.step("y", t / d, "t / d"), c.lines


def gelu_erf(t: Q, dtype: str):
    c = Chain(dtype)
    c3 = c.step("c3", Q(1 / math.sqrt(2)), "1 / sqrt 2")
    s = c.step("s", c3 * t, "c3 * t")
    e = c.step("e", erf_q(s), "erf(s)")
    d = c.step("d", 1 + e, "1 + e")
    p = c.step("p", t * d, "t * d")
    return c.step("y", p / 2, "0.5 * p"), c.lines


CASES = {
    "epilogue_silu.txt": [("f16", "silu", Q(5, 256)), ("f16", "silu", Q(-3, 2)), ("bf16", "silu", Q(1))],
    "epilogue_gelu.txt": [("f16", "gelu_tanh", Q(1)), ("f16", "gelu_erf", Q(-1, 2)),
                          ("bf16", "gelu_erf", Q(2)), ("bf16", "gelu_tanh", Q(-3, 4))],
}
OPS = {"silu": silu, "gelu_tanh": gelu_tanh, "gelu_erf": gelu_erf}


def derive(fixture: str):
    """(comment lines, "case <dtype> <op> <t> <y>" lines) of one fixture."""
    comments, cases = [], []
    for dtype, op, t in CASES[fixture]:
        y, lines = OPS[op](t, dtype)
        comments.append(f"# {dtype} {op.upper()} at t = {float(t)!r}")
        comments.extend(lines)
        comments.append("#")
        cases.append(f"case {dtype} {op} {float(t)!r} {float(y)!r}")
    return comments, cases


if __name__ == "__main__":
    for fixture in CASES:
        comments, cases = derive(fixture)
        print(f"# ---- {fixture}")
        print("\n".join(comments))
        print("\n".join(cases))
