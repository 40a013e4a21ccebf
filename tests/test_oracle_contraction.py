"""Pins of the widened oracle (oracle/oracle_contraction.c) against what the
pages and the mathematics fix, without a GPU.

* binary64 -> binary16 / bfloat16 rounding: exact rational rounding (tests/
  exact.py), the already pinned binary32 -> binary16 conversion, and the
  round-to-nearest-even bit formula for bfloat16;
* epilogue chains: the hand-worked cases under tests/golden/ (each
  primitive rounds: "ML compiler internals", ContractionEpilogue row and
  section "SwiGLU and GeLU FFN"), closed forms at 0 and at large |t|, and
  the rounding-error bound of the chain around the exact function;
* the contraction: the binary16 head against the base oracle, exact
  integer cases for the bias, the extra operands, the FP32 output and the
  bfloat16 head (sums exact, so only the stated roundings remain).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import exact


def _chain(t_vals, op, dtype, mutation=0):
    bits = exact.float_to_bits(np.asarray(t_vals, dtype=np.float64), dtype).reshape(1, -1)
    y = oracle.epilogue(bits, None, dtype=dtype, steps=[op], mutation=mutation)
    return _decode(y.ravel(), dtype)


def _decode(bits, dtype):
    bits = np.asarray(bits, dtype=np.uint16)
    return bits.view(np.float16).astype(np.float64) if dtype == "f16" else exact.bf16_bits_to_float(bits)


# ---- roundings --------------------------------------------------------------------
def test_f64_to_f16_equals_the_pinned_binary32_conversion():
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    got = oracle.f64_to_f16_rn(f.astype(np.float64))
    want = oracle.f32_to_f16_rn(f)
    assert np.array_equal(got, want)


def _ties_and_neighbours(fmt):
    """Midpoints between consecutive finite values (ties) and values just off them."""
    if fmt == "f16":
        vals = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    else:
        vals = exact.bf16_bits_to_float(np.arange(0, 0x7F80, 7, dtype=np.uint16))
    mids = (vals[:-1] + vals[1:]) / 2           # exact in binary64
    out = np.concatenate([mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf)])
    return np.concatenate([out, -out])


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_f64_rounding_against_exact_rationals(fmt):
    rng = np.random.default_rng(12)
    cand = _ties_and_neighbours(fmt)
    sample = np.concatenate([rng.choice(cand, 3000, replace=False),
                             rng.standard_normal(1500) * 10.0 ** rng.integers(-9, 6, 1500),
                             [65504.0, 65519.99, 65520.0, 3.38e38, 3.3961e38, 3.3963e38, 2.0 ** -24,
                              2.0 ** -25, 2.0 ** -133, 2.0 ** -134, 1.5 * 2.0 ** -134]])
    conv = oracle.f64_to_f16_rn if fmt == "f16" else oracle.f64_to_bf16_rn
    got = _decode(conv(sample), fmt)
    want = np.array([exact.rn_format(Fraction(float(v)), fmt) for v in sample])
    assert exact.same_values(got, want)


def test_bf16_rounding_matches_the_bit_formula():
    # round to nearest even on the upper 16 bits of a binary32: add 0x7FFF
    # plus the lowest kept bit, then truncate (finite inputs)
    rng = np.random.default_rng(13)
    u = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    keep = np.isfinite(f)
    u, f = u[keep], f[keep]
    want = ((u.astype(np.uint64) + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    got = oracle.f64_to_bf16_rn(f.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_decode_is_the_upper_half_of_binary32():
    h = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f32(h)
    want = (h.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ---- epilogue chains --------------------------------------------------------------
@pytest.mark.parametrize("name", ["epilogue_silu.txt", "epilogue_gelu.txt"])
def test_stored_chains_are_what_the_derivation_script_writes(name):
    # the fixtures' values come from tests/golden/derive_epilogue_chains.py,
    # which imports neither the oracle nor the CUDA package
    import importlib.util
    path = os.path.join(os.path.dirname(__file__), "golden", "derive_epilogue_chains.py")
    spec = importlib.util.spec_from_file_location("derive_epilogue_chains", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    _, cases = mod.derive(name)
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as fh:
        stored = [ln.strip() for ln in fh if ln.startswith("case ")]
    assert cases == stored


@pytest.mark.parametrize("name", ["epilogue_silu.txt", "epilogue_gelu.txt"])
def test_worked_chains(name):
    for dtype, op, t, y in exact.parse_chain_golden(name):
        got = _chain([t], op, dtype)[0]
        assert got == y, (dtype, op, t, got, y)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_chain_closed_forms(dtype):
    for op in ("silu", "gelu_tanh", "gelu_erf"):
        z = _chain([0.0], op, dtype)[0]
        assert z == 0.0, (op, dtype)
        big = _chain([16.0, 64.0], op, dtype)                 # sigmoid / erf saturate at 1
        assert np.array_equal(big, [16.0, 64.0]), (op, dtype, big)
        neg = _chain([-64.0], op, dtype)[0]                    # far left tail: a zero (or tiny for bf16)
        assert abs(neg) < 2.0 ** -20, (op, dtype, neg)
    # binary16: exp(20) overflows to infinity, so d = inf and silu(-20) = -0
    if dtype == "f16":
        y = _chain([-20.0], "silu", "f16")[0]
        assert y == 0.0 and math.copysign(1.0, y) < 0


def _silu(t):
    return t / (1.0 + math.exp(-t))


def _gelu_tanh(t):
    return 0.5 * t * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (t + 0.044715 * t ** 3)))


def _gelu_erf(t):
    return 0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0)))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("op,fn,k", [("silu", _silu, 4), ("gelu_tanh", _gelu_tanh, 12), ("gelu_erf", _gelu_erf, 6)])
def test_chain_within_its_rounding_error_bound(dtype, op, fn, k):
    # each of the chain's roundings adds at most one unit roundoff u; k
    # bounds how many reach the result (with the rounded constants of the
    # tanh form included), so |y - f(t)| <= k u (|t| + |f(t)|) + tiny
    u = 2.0 ** -11 if dtype == "f16" else 2.0 ** -8
    rng = np.random.default_rng(14)
    t = rng.uniform(-6, 6, 4000)
    t = _decode(exact.float_to_bits(np.array([exact.rn_format(Fraction(v), dtype) for v in t]), dtype), dtype)
    y = _chain(t, op, dtype)
    f = np.array([fn(v) for v in t])
    assert np.all(np.abs(y - f) <= k * u * (np.abs(t) + np.abs(f)) + 2.0 ** -24)


# ---- the contraction --------------------------------------------------------------
def _smallint(rng, shape, lo=-4, hi=5):
    return rng.integers(lo, hi, size=shape).astype(np.float64)


def test_f16_head_with_bias_is_the_base_oracle():
    rng = np.random.default_rng(15)
    x = rng.standard_normal((37, 300)).astype(np.float16)
    w = (rng.standard_normal((29, 300)) * 0.05).astype(np.float16)
    b = (rng.standard_normal(29) * 0.1).astype(np.float16)
    y, p = oracle.contraction(x, w, b, want_proj=True)
    y0, p0 = oracle.linear_f16(x, w, b, want_proj=True)
    assert np.array_equal(y, y0) and np.array_equal(p, p0)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_exact_integer_chain(dtype):
    # small integers: every sum, bias add, addend and multiplier is exact,
    # so y = ((S + b) * m + r) with no rounding at all
    rng = np.random.default_rng(16)
    M, N, K = 6, 5, 9
    x, w, b = _smallint(rng, (M, K)), _smallint(rng, (N, K)), _smallint(rng, N)
    m = 2.0 ** rng.integers(-2, 3, size=(M, N))          # powers of two, not symmetric
    r = _smallint(rng, (M, N))
    bits = lambda a: exact.float_to_bits(a, dtype)
    y = oracle.contraction(bits(x), bits(w), bits(b), dtype=dtype,
                           steps=[("mul", bits(m)), ("add", bits(r))])
    want = ((x @ w.T) + b) * m + r
    assert np.array_equal(_decode(y.ravel(), dtype).reshape(M, N), want)
    # adding the negated head value gives +0; multiplying by one changes nothing
    y2 = oracle.contraction(bits(x), bits(w), None, dtype=dtype, steps=[("add", bits(-(x @ w.T)))])
    assert np.all(_decode(y2.ravel(), dtype) == 0.0)
    y3 = oracle.contraction(bits(x), bits(w), bits(b), dtype=dtype, steps=[("mul", bits(np.ones((M, N))))])
    assert np.array_equal(_decode(y3.ravel(), dtype).reshape(M, N), (x @ w.T) + b)


def test_no_bias_is_the_rounded_sum():
    rng = np.random.default_rng(17)
    x = rng.standard_normal((8, 64)).astype(np.float16)
    w = rng.standard_normal((8, 64)).astype(np.float16)
    y, p = oracle.contraction(x, w, None, want_proj=True)
    assert np.array_equal(y, p)


def test_f32_output_exact_for_integers_and_within_the_sum_bound():
    rng = np.random.default_rng(18)
    M, N, K = 7, 6, 40
    x, w, b = _smallint(rng, (M, K)), _smallint(rng, (N, K)), _smallint(rng, N)
    y = oracle.contraction(x.astype(np.float16), w.astype(np.float16), b.astype(np.float16), out_f32=True)
    assert y.dtype == np.float32 and np.array_equal(y.astype(np.float64), x @ w.T + b)
    # sums that round: within gamma_K sum|x w| of the exact sum (Higham, section 3.1)
    xr = rng.standard_normal((M, K)).astype(np.float16)
    wr = rng.standard_normal((N, K)).astype(np.float16)
    y = oracle.contraction(xr, wr, None, out_f32=True).astype(np.float64)
    S, A = exact.exact_sums(xr.view(np.uint16), wr.view(np.uint16))
    u = 2.0 ** -24
    gamma = K * u / (1 - K * u)
    for mm in range(M):
        for nn in range(N):
            assert abs(Fraction(float(y[mm, nn])) - S[mm][nn]) <= Fraction(gamma) * A[mm][nn]


def test_bf16_head_rounds_to_bfloat16():
    # integer sums beyond 256 are not all bfloat16 numbers (8 significand
    # bits): the head value is the exact sum rounded to bfloat16
    rng = np.random.default_rng(19)
    M, N, K = 5, 4, 64
    x, w = _smallint(rng, (M, K), -8, 9), _smallint(rng, (N, K), -8, 9)
    b = _smallint(rng, N)
    bits = lambda a: exact.float_to_bits(a, "bf16")
    y, p = oracle.contraction(bits(x), bits(w), bits(b), dtype="bf16", want_proj=True)
    S = x @ w.T
    want_p = np.array([[exact.rn_format(Fraction(float(v)), "bf16") for v in row] for row in S])
    want_y = np.array([[exact.rn_format(Fraction(want_p[i, j]) + Fraction(float(b[j])), "bf16")
                        for j in range(N)] for i in range(M)])
    assert np.array_equal(exact.bf16_bits_to_float(p.ravel()).reshape(M, N), want_p)
    assert np.array_equal(exact.bf16_bits_to_float(y.ravel()).reshape(M, N), want_y)
    assert np.any(want_p != S)  # the case does exercise the rounding


def test_steps_apply_in_order():
    rng = np.random.default_rng(20)
    x = rng.standard_normal((4, 32)).astype(np.float16)
    w = rng.standard_normal((6, 32)).astype(np.float16)
    m = np.full((4, 6), 3.0, dtype=np.float16)
    a = oracle.contraction(x, w, None, steps=["silu", ("mul", m)])
    bb = oracle.contraction(x, w, None, steps=[("mul", m), "silu"])
    assert not np.array_equal(a, bb)


# ---- the pins have teeth ----------------------------------------------------------
NEW_MUTATIONS = {
    11: "binary64 rounding truncates",
    12: "SiLU rounded once instead of per primitive",
    13: "GELU (erf form) without the factor 0.5",
    14: "multiplier read transposed",
    15: "bfloat16 head rounded as binary16",
}


def _new_pins_pass(mutation):
    for name in ("epilogue_silu.txt", "epilogue_gelu.txt"):
        for dtype, op, t, y in exact.parse_chain_golden(name):
            if _chain([t], op, dtype, mutation=mutation)[0] != y:
                return False
    ties = _ties_and_neighbours("f16")[:2000]
    got = _decode(oracle.f64_to_f16_rn(ties, mutation=mutation), "f16")
    if not exact.same_values(got, [exact.rn_format(Fraction(float(v)), "f16") for v in ties]):
        return False
    rng = np.random.default_rng(21)
    M, N, K = 5, 4, 64
    for dtype in ("f16", "bf16"):
        x, w = _smallint(rng, (M, K), -8, 9), _smallint(rng, (N, K), -8, 9)
        m = 2.0 ** rng.integers(-2, 3, size=(M, N))
        bits = lambda a: exact.float_to_bits(a, dtype)
        y = oracle.contraction(bits(x), bits(w), None, dtype=dtype, steps=[("mul", bits(m))], mutation=mutation)
        S = x @ w.T
        want = np.array([[exact.rn_format(Fraction(float(v)), dtype) for v in row] for row in S]) * m
        want = np.array([[exact.rn_format(Fraction(float(v)), dtype) for v in row] for row in want])
        if not np.array_equal(_decode(y.ravel(), dtype).reshape(M, N), want):
            return False
    return True


def test_unmutated_widened_oracle_passes_its_pins():
    assert _new_pins_pass(0)


@pytest.mark.parametrize("mutation", sorted(NEW_MUTATIONS))
def test_widened_oracle_planted_mistake_is_caught(mutation):
    assert not _new_pins_pass(mutation), NEW_MUTATIONS[mutation]


# ---- grouped ----------------------------------------------------------------------
def test_grouped_is_the_diagonal_of_one_contraction():
    # all groups' rows against all groups' W blocks in one contraction: block
    # (g, g) of the result is group g of the grouped contraction
    rng = np.random.default_rng(22)
    G, M, N, K = 3, 5, 4, 24
    x = rng.standard_normal((G, M, K)).astype(np.float16)
    w = rng.standard_normal((G * N, K)).astype(np.float16)
    b = rng.standard_normal(G * N).astype(np.float16)
    r = rng.standard_normal((G, M, N)).astype(np.float16)
    grouped = oracle.contraction_grouped(x, w, b, steps=[("mul", r), "silu"])
    full_r = np.zeros((G * M, G * N), dtype=np.float16)
    for g in range(G):
        full_r[g * M:(g + 1) * M, g * N:(g + 1) * N] = r[g]
    full = oracle.contraction(x.reshape(G * M, K), w, b, steps=[("mul", full_r), "silu"])
    for g in range(G):
        assert np.array_equal(grouped[g], full[g * M:(g + 1) * M, g * N:(g + 1) * N])
