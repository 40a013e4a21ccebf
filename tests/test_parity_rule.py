"""The comparison rule itself (tests/parity.py), on the CPU.

The legal interval must contain the oracle's own result and results of
other FP32 summation orders, and the rule must reject what a plausible bug
produces (a dropped term, the bias added before rounding).
"""
import numpy as np
import torch

import oracle
from linear_fp16_gb300 import synth
from tests.parity import U_RN, check_rows, compare, intervals, legal_interval


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _other_order(x, w, b):
    # a legal FP32 order: 16-term pairwise blocks, blocks summed in sequence
    xf, wf = x.float().numpy(), w.float().numpy()
    acc = np.zeros((xf.shape[0], wf.shape[0]), np.float32)
    for k0 in range(0, xf.shape[1], 16):
        blk = (xf[:, None, k0:k0 + 16] * wf[None, :, k0:k0 + 16]).astype(np.float32)
        while blk.shape[2] > 1:
            if blk.shape[2] % 2:
                blk = np.concatenate([blk, np.zeros_like(blk[:, :, :1])], axis=2)
            blk = (blk[:, :, 0::2] + blk[:, :, 1::2]).astype(np.float32)
        acc = (acc + blk[:, :, 0]).astype(np.float32)
    return (acc.astype(np.float16).astype(np.float32) + b.float().numpy()[None, :]).astype(np.float16)


def test_interval_holds_oracle_and_another_order():
    x, w, b = synth.make_inputs(64, 96, 1000, "normal", 3)
    lo, hi = legal_interval(x.numpy(), w.numpy(), b.numpy())
    yr, pr = oracle.linear_f16(_bits(x), _bits(w), _bits(b), want_proj=True)
    for y in (yr.view(np.float16), _other_order(x, w, b)):
        v = y.astype(np.float64)
        assert np.all((v >= lo) & (v <= hi))
        ok, rep = compare(y.view(np.uint16), yr, pr, exact=False, interval=(lo, hi))
        assert ok, rep


def test_rule_rejects_a_dropped_term():
    x, w, b = synth.make_inputs(32, 48, 256, "normal", 4)
    yr, pr = oracle.linear_f16(_bits(x), _bits(w), _bits(b), want_proj=True)
    iv = legal_interval(x.numpy(), w.numpy(), b.numpy())
    dropped = oracle.linear_f16(_bits(x), _bits(w), _bits(b), mutation=3)
    ok, rep = compare(dropped, yr, pr, exact=False, interval=iv)
    assert not ok and rep["beyond_2ulp_inside_interval"] < rep["beyond_2ulp"]


def test_bias_before_rounding_needs_the_exact_cases():
    # Adding b before rounding moves y by at most one ulp, which no 2-ulp
    # rule can see; the bit-exact cases (small integers, the golden
    # fixtures) are what catch it.
    x, w, b = synth.make_inputs(32, 48, 256, "uniform", 5)
    x = x * 64
    yr, pr = oracle.linear_f16(_bits(x), _bits(w), _bits(b), want_proj=True)
    early = oracle.linear_f16(_bits(x), _bits(w), _bits(b), mutation=1)
    ok, _ = compare(early, yr, pr, exact=False, interval=legal_interval(x.numpy(), w.numpy(), b.numpy()))
    assert ok
    from tests import exact as ex
    xg, wg, bg, _ = ex.parse_golden("round_before_bias.txt")
    yg = oracle.linear_f16(xg, wg, bg)
    eg = oracle.linear_f16(xg, wg, bg, mutation=1)
    ok, _ = compare(eg, yg, None, exact=True)
    assert not ok


def test_exact_mode_is_bitwise():
    yr = np.array([[0x3c00, 0x0000]], np.uint16)
    ok, _ = compare(np.array([[0x3c00, 0x8000]], np.uint16), yr, None, exact=True)
    assert ok  # +0 == -0
    ok, _ = compare(np.array([[0x3c01, 0x0000]], np.uint16), yr, None, exact=True)
    assert not ok


def test_ieee_interval_holds_round_to_nearest_orders():
    # u = 2^-24 bounds every round-to-nearest FP32 order: the oracle's own
    # sequential sum and a pairwise one both lie inside it, and it nests in
    # the wider interval that also admits truncation
    x, w, b = synth.make_inputs(48, 80, 2000, "normal", 6)
    (lo, hi), (lo_t, hi_t) = intervals(x.numpy(), w.numpy(), b.numpy())
    assert np.all(lo_t <= lo) and np.all(hi <= hi_t)
    assert np.array_equal(np.stack(legal_interval(x.numpy(), w.numpy(), b.numpy())), np.stack((lo, hi)))
    assert np.array_equal(np.stack(legal_interval(x.numpy(), w.numpy(), b.numpy(), u=U_RN)), np.stack((lo, hi)))
    yr, pr = oracle.linear_f16(_bits(x), _bits(w), _bits(b), want_proj=True)
    for y in (yr.view(np.float16), _other_order(x, w, b)):
        v = y.astype(np.float64)
        assert np.all((v >= lo) & (v <= hi))
        ok, rep = compare(y.view(np.uint16), yr, pr, exact=False, interval=(lo, hi), wide_interval=(lo_t, hi_t))
        assert ok and rep["beyond_2ulp_outside_interval"] == 0, rep
        assert rep["beyond_2ulp_outside_truncating_interval"] == 0, rep


def test_check_rows_matches_compare_and_counts_strict_ulps():
    x, w, b = synth.make_inputs(40, 64, 512, "normal", 7)
    yr, pr = oracle.linear_f16(_bits(x), _bits(w), _bits(b), want_proj=True)
    rows = np.array([0, 3, 17, 39])
    ok, rep = check_rows(yr[rows], _bits(x), _bits(w), _bits(b), exact=False, rows=rows)
    assert ok and rep["bad"] == 0 and rep["beyond_2ulp_of_y"] == 0 and rep["max_ulps_of_y"] == 0
    # a planted 3-ulp error in one element: beyond 2 ulps, outside both intervals
    bad = yr[rows].copy()
    bad[1, 5] = np.uint16(int(bad[1, 5]) + 3) if (bad[1, 5] & 0x7c00) != 0x7c00 else bad[1, 5]
    ok, rep = check_rows(bad, _bits(x), _bits(w), _bits(b), exact=False, rows=rows)
    assert not ok and rep["beyond_2ulp_of_y"] == 1 and rep["beyond_2ulp_outside_interval"] == 1
    # the dropped-term mutation fails through check_rows too
    dropped = oracle.linear_f16(_bits(x), _bits(w), _bits(b), mutation=3)
    ok, rep = check_rows(dropped, _bits(x), _bits(w), _bits(b), exact=False)
    assert not ok
