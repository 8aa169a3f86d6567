"""Pins of the oracle's scale step (CPU only).

The oracle computes the scale in IEEE fp32 (one division of the floored
amax by the format maximum) and, in the power-of-two modes, rounds the fp32
ratio up to 2^k with frexpf.  These tests check it against exact rational
arithmetic over every positive finite BF16 amax, and against the hand-worked
special values in tests/golden/scale_specials.txt.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bruteforce import F32_1E4, FMT_MAX, pow2_ceil_exponent, rn_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scale_specials.txt")
FMTS = [("e4m3", oracle.FMT_E4M3), ("e2m1", oracle.FMT_E2M1)]


def positive_bf16_amax():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)   # +0 .. largest finite
    return (bits << 16).view(np.float32)


def test_floor_constant():
    assert np.float32(1e-4).view(np.uint32) == 0x38D1B717
    assert F32_1E4 == float(np.float32(1e-4))


@pytest.mark.parametrize("name,fmt", FMTS)
def test_fp32_scale_is_correctly_rounded_quotient(name, fmt):
    a = positive_bf16_amax()
    s, e = oracle.scale(a, fmt, oracle.SCALE_FP32)
    assert np.all(e == -1)
    for ai, si in zip(a[::7].tolist(), s[::7].tolist()):
        want = rn_f32(Fraction(max(ai, F32_1E4)) / Fraction(FMT_MAX[name]))
        assert si == want, (ai, si, want)


@pytest.mark.parametrize("name,fmt", FMTS)
@pytest.mark.parametrize("mode", [oracle.SCALE_FP32_POW2, oracle.SCALE_UE8M0])
def test_pow2_scale_is_smallest_power_of_two_above_exact_ratio(name, fmt, mode):
    """Every BF16 amax: the oracle ceils the fp32-rounded ratio; the exact
    rational ratio gives the same power of two (the two readings agree)."""
    a = positive_bf16_amax()
    s, e = oracle.scale(a, fmt, mode)
    for ai, si, ei in zip(a.tolist(), s.tolist(), e.tolist()):
        k = pow2_ceil_exponent(Fraction(max(ai, F32_1E4)) /
                               Fraction(FMT_MAX[name]))
        assert ei == k + 127, (ai, ei, k)
        assert si == 2.0 ** k


@pytest.mark.parametrize("name,fmt", FMTS)
def test_pow2_bracket(name, fmt):
    """s/2 < max(amax,1e-4)/fmt_max <= s for every BF16 amax."""
    a = positive_bf16_amax().astype(np.float64)
    s, _ = oracle.scale(a.astype(np.float32), fmt, oracle.SCALE_UE8M0)
    r = np.maximum(a, F32_1E4) / FMT_MAX[name]
    assert np.all(r <= s) and np.all(r > s.astype(np.float64) / 2)


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        bits, fmt, sbits, ue8m0 = line.split()[:4]
        rows.append((int(bits, 16), fmt, sbits, int(ue8m0)))
    return rows


@pytest.mark.parametrize("bits,name,sbits,ue8m0", _golden_rows())
def test_golden_specials(bits, name, sbits, ue8m0):
    fmt = oracle.FMT_E4M3 if name == "e4m3" else oracle.FMT_E2M1
    amax = (np.array([bits], np.uint32) << 16).view(np.float32)
    s, _ = oracle.scale(amax, fmt, oracle.SCALE_FP32)
    if sbits != "-":
        assert s.view(np.uint32)[0] == int(sbits, 16)
    _, e = oracle.scale(amax, fmt, oracle.SCALE_UE8M0)
    assert e[0] == ue8m0
    s2, _ = oracle.scale(amax, fmt, oracle.SCALE_FP32_POW2)
    assert s2[0] == np.float32(2.0 ** (ue8m0 - 127))
