"""Pins of the oracle's binary16 <-> binary32 conversions.

The oracle writes RN16 from the IEEE 754 definition.  These tests compare it
with independent implementations: numpy's float16 casts, the C compiler's
_Float16 cast (exhaustive over all 2^32 inputs), and the exact-rational
rounding in tests/exact.py.
"""
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import exact

HERE = os.path.dirname(os.path.abspath(__file__))


def test_f16_to_f32_all_65536_patterns():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    mine = oracle.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    same = (mine.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(mine) & np.isnan(ref))
    assert same.all(), np.flatnonzero(~same)[:10]
    # and against the exact decoding from the bit fields
    for bits in list(range(0, 2048, 7)) + [0x0001, 0x03ff, 0x0400, 0x7bff, 0x8001, 0xfbff]:
        assert Fraction(float(mine[bits])) == exact.f16_bits_to_fraction(bits)


def _special_f32_patterns():
    pats = []
    # every binary16 value, the midpoints between neighbours, and one float
    # ulp either side of each midpoint: the places where RN16 decides
    h = np.arange(0, 0x7c00, dtype=np.uint32).astype(np.uint16)
    v = h.view(np.float16).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2
    for arr in (v, mids):
        f = arr.astype(np.float32)
        pats.append(f.view(np.uint32))
        pats.append(np.nextafter(f, np.float32(np.inf)).view(np.uint32))
        pats.append(np.nextafter(f, np.float32(0)).view(np.uint32))
    pats.append(np.array([0x477fefff, 0x477ff000, 0x477ff001, 0x7f7fffff, 0x00000001,
                          0x33000000, 0x33000001, 0x337fffff, 0x7f800000, 0x7fc00000],
                         dtype=np.uint32))
    allp = np.concatenate(pats)
    return np.concatenate([allp, allp | np.uint32(0x80000000)])


def test_f32_to_f16_rounding_boundaries_vs_numpy():
    u = _special_f32_patterns()
    f = u.view(np.float32)
    mine = oracle.f32_to_f16_rn(f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.isnan(mine[nan].view(np.float16)).all()


def test_f32_to_f16_random_vs_numpy():
    rng = np.random.default_rng(12345)
    u = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    mine = oracle.f32_to_f16_rn(f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_f32_to_f16_vs_exact_rational():
    rng = np.random.default_rng(7)
    # magnitudes across the subnormal, normal and overflow ranges
    e = rng.integers(-30, 18, size=3000)
    m = rng.random(3000) + 1.0
    f = (np.sign(rng.random(3000) - 0.5) * m * np.exp2(e)).astype(np.float32)
    mine = oracle.f32_to_f16_rn(f).view(np.float16).astype(np.float64)
    for fv, mv in zip(f, mine):
        assert exact.rn16(Fraction(float(fv))) == mv or (fv == 0)


@pytest.mark.slow
def test_f32_to_f16_exhaustive_vs_compiler(tmp_path):
    so = oracle.build()
    exe = str(tmp_path / "f16_exhaustive")
    subprocess.run(["gcc", "-O2", "-std=c11", "-pthread", os.path.join(HERE, "f16_exhaustive.c"),
                    so, "-o", exe, f"-Wl,-rpath,{os.path.dirname(so)}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout
