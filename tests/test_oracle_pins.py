"""Pins of the oracle's linear op against what the pages and mathematics fix.

* tests/golden/: hand-worked examples of the two contract rules ("Tensor
  Programs, Part 1", section "One Program and One Numerical Contract") and of
  the IEEE rounding edges (overflow, gradual underflow).
* brute force on tiny shapes against exact rational arithmetic: bit-exact
  when every FP32 partial sum is exact (small integers), and inside the
  Higham error interval otherwise.
* closed forms: identity and permutation weights, x = 0, zero bias.
* invariants: sign symmetry, power-of-two scaling, row/column permutation,
  independence of the thread count.
"""
import numpy as np
import pytest

import oracle
from tests import exact

GOLDENS = ["round_before_bias.txt", "fp32_accumulation.txt", "no_product_rounding.txt",
           "overflow_boundary.txt", "subnormal_rounding.txt"]


def _y(x, w, b, **kw):
    return oracle.linear_f16(x, w, b, **kw).view(np.float16).astype(np.float64)


@pytest.mark.parametrize("name", GOLDENS)
def test_golden(name):
    x, w, b, y = exact.parse_golden(name)
    got = _y(x, w, b)
    assert exact.same_values(got, y), (name, got, y)


def _rand_f16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def _small_ints(rng, shape, lo=-4, hi=4):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float16)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 5), (3, 2, 7), (4, 4, 16), (1, 5, 33), (5, 1, 9)])
def test_small_integers_exact(M, N, K):
    # |S| <= 16 K < 2^24: every partial sum in any order is exact in FP32,
    # so the contract fixes y exactly: RN16(RN16(S) + b).
    rng = np.random.default_rng(100 + M * 100 + N * 10 + K)
    x, w, b = _small_ints(rng, (M, K)), _small_ints(rng, (N, K)), _small_ints(rng, (N,))
    want = exact.exact_linear(x.view(np.uint16), w.view(np.uint16), b.view(np.uint16))
    assert exact.same_values(_y(x, w, b), want)


def test_dyadic_exact_with_rounding_in_both_steps():
    # Values with few significant bits: every FP32 partial sum is exact but
    # both binary16 roundings are exercised (sums need up to ~20 bits).
    rng = np.random.default_rng(5)
    M, N, K = 6, 7, 12
    x = (rng.integers(-63, 64, size=(M, K)) * 2.0 ** rng.integers(-3, 4, size=(M, K))).astype(np.float16)
    w = (rng.integers(-63, 64, size=(N, K)) * 2.0 ** rng.integers(-3, 4, size=(N, K))).astype(np.float16)
    b = (rng.integers(-1023, 1024, size=N) * 2.0 ** -5).astype(np.float16)
    want = exact.exact_linear(x.view(np.uint16), w.view(np.uint16), b.view(np.uint16))
    assert exact.same_values(_y(x, w, b), want)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_inside_higham_interval(seed):
    rng = np.random.default_rng(seed)
    M, N, K = 4, 5, 24
    x, w, b = _rand_f16(rng, (M, K)), _rand_f16(rng, (N, K), 0.5), _rand_f16(rng, (N,), 0.1)
    lo, hi = exact.higham_interval(x.view(np.uint16), w.view(np.uint16), b.view(np.uint16))
    got = _y(x, w, b)
    assert np.all(lo <= got) and np.all(got <= hi)


def test_identity_weight_closed_form():
    # W = I (N = K): y = RN16(x + b), computed here by numpy's float16 add
    rng = np.random.default_rng(11)
    M, K = 9, 16
    x = _rand_f16(rng, (M, K), 3.0)
    b = _rand_f16(rng, (K,), 0.01)
    w = np.eye(K, dtype=np.float16)
    want = (x.astype(np.float32) + b.astype(np.float32)).astype(np.float16)
    assert exact.same_values(_y(x, w, b), want.astype(np.float64))


def test_permutation_weight_closed_form():
    rng = np.random.default_rng(12)
    M, K = 7, 13
    perm = rng.permutation(K)
    w = np.eye(K, dtype=np.float16)[perm]          # row n selects x[:, perm[n]]
    x = _rand_f16(rng, (M, K), 10.0)
    b = _rand_f16(rng, (K,), 1.0)
    want = (x[:, perm].astype(np.float32) + b.astype(np.float32)).astype(np.float16)
    assert exact.same_values(_y(x, w, b), want.astype(np.float64))


def test_zero_input_gives_bias():
    rng = np.random.default_rng(13)
    b = _rand_f16(rng, (10,))
    got = _y(np.zeros((3, 6), np.float16), _rand_f16(rng, (10, 6)), b)
    assert exact.same_values(got, np.broadcast_to(b.astype(np.float64), (3, 10)))


def test_zero_k_gives_bias():
    b = np.array([1.5, -2.0, -0.0], np.float16)
    got = oracle.linear_f16(np.zeros((2, 0), np.float16), np.zeros((3, 0), np.float16), b)
    vals = got.view(np.float16).astype(np.float64)
    assert exact.same_values(vals, np.broadcast_to(b.astype(np.float64), (2, 3)))
    # S = +0; +0 + (-0) = +0 under round-to-nearest
    assert np.all(got[:, 2] == 0x0000)


def test_zero_bias_gives_rounded_projection():
    rng = np.random.default_rng(14)
    x, w = _rand_f16(rng, (5, 40)), _rand_f16(rng, (6, 40))
    y, p = oracle.linear_f16(x, w, np.zeros(6, np.float16), want_proj=True)
    assert exact.same_values(y.view(np.float16), p.view(np.float16))


def test_sign_symmetry():
    rng = np.random.default_rng(15)
    x, w, b = _rand_f16(rng, (8, 50)), _rand_f16(rng, (9, 50)), _rand_f16(rng, (9,))
    y = _y(x, w, b)
    assert exact.same_values(_y(-x, w, -b), -y)
    assert exact.same_values(_y(x, -w, -b), -y)


def test_power_of_two_scaling():
    rng = np.random.default_rng(16)
    x, w = _rand_f16(rng, (8, 50)), _rand_f16(rng, (9, 50))
    zb = np.zeros(9, np.float16)
    y = _y(x, w, zb)
    for s in (-3, 2, 4):
        assert exact.same_values(_y((x.astype(np.float32) * 2.0 ** s).astype(np.float16), w, zb),
                                 y * 2.0 ** s)


def test_row_and_column_permutations():
    rng = np.random.default_rng(17)
    M, N, K = 11, 12, 30
    x, w, b = _rand_f16(rng, (M, K)), _rand_f16(rng, (N, K)), _rand_f16(rng, (N,))
    y = _y(x, w, b)
    pm, pn = rng.permutation(M), rng.permutation(N)
    assert exact.same_values(_y(x[pm], w, b), y[pm])
    assert exact.same_values(_y(x, w[pn], b[pn]), y[:, pn])


def test_thread_count_does_not_change_result():
    rng = np.random.default_rng(18)
    x, w, b = _rand_f16(rng, (37, 64)), _rand_f16(rng, (21, 64)), _rand_f16(rng, (21,))
    ref = oracle.linear_f16(x, w, b, nthreads=1)
    for t in (2, 3, 8, 64):
        assert np.array_equal(oracle.linear_f16(x, w, b, nthreads=t), ref)


def test_config_shape_smallint_is_exact_on_a_slice():
    # the exactness config's value ranges: |S| <= 770*16 < 2^24, so the
    # oracle equals the exact contract on it; checked on a few rows
    rng = np.random.default_rng(19)
    x, w, b = _small_ints(rng, (3, 770)), _small_ints(rng, (5, 770)), _small_ints(rng, (5,))
    want = exact.exact_linear(x.view(np.uint16), w.view(np.uint16), b.view(np.uint16))
    assert exact.same_values(_y(x, w, b), want)
