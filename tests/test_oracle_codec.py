"""Pins of the oracle's E4M3 / E2M1 encoders (CPU only).

The oracle encodes with bit arithmetic; these tests compare it with a
value-space nearest-code search (tests/bruteforce.py) that follows the OCP
format definitions directly.
"""
import numpy as np
import pytest

import oracle
from bruteforce import decode, decode_table, nearest_code

FMTS = [("e4m3", oracle.FMT_E4M3), ("e2m1", oracle.FMT_E2M1)]


def all_finite_bf16_as_f32():
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)]


def test_decode_table_facts():
    # OCP facts: E4M3FN has 126 finite nonzero magnitudes, max 448, min
    # subnormal 2^-9, min normal 2^-6; E2M1 magnitudes 0..6.
    t = decode_table("e4m3")
    assert t.size == 127 and t[-1] == 448.0 and t[1] == 2.0 ** -9
    assert t[8] == 2.0 ** -6 and np.all(np.diff(t) > 0)
    assert list(decode_table("e2m1")) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


@pytest.mark.parametrize("name,fmt", FMTS)
def test_exhaustive_bf16(name, fmt):
    """Every finite BF16 bit pattern (65,536 minus NaN/Inf), unscaled."""
    q = all_finite_bf16_as_f32()
    got = oracle.encode(q, fmt)
    want = nearest_code(q, name)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (q[bad[:5]], got[bad[:5]], want[bad[:5]])


def _neighbourhood(points, ulps):
    p = np.asarray(points, dtype=np.float32)
    out = [p]
    up, dn = p.copy(), p.copy()
    for _ in range(ulps):
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(-np.inf))
        out += [up, dn]
    return np.concatenate(out)


@pytest.mark.parametrize("name,fmt", FMTS)
def test_midpoints_and_neighbours(name, fmt):
    """Every rounding boundary of the format, +-4 fp32 ulps, both signs."""
    t = decode_table(name)
    mids = (t[:-1] + t[1:]) / 2
    extra = [t[-1], t[-1] * 1.0001, t[-1] * 1.05, 1e30, 3.0e38, 1e-30, 1e-42]
    pts = _neighbourhood(np.concatenate([mids, t, extra]), 4)
    pts = np.concatenate([pts, -pts])
    got = oracle.encode(pts, fmt)
    want = nearest_code(pts, name)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("name,fmt", FMTS)
def test_random_fp32_patterns(name, fmt):
    """4M random fp32 bit patterns covering the format's range and beyond."""
    rng = np.random.default_rng(1234)
    lo = np.float32(2.0 ** -14).view(np.uint32)
    hi = np.float32(1024.0).view(np.uint32)
    bits = rng.integers(lo, hi, size=1 << 22, dtype=np.uint32)
    bits |= (rng.integers(0, 2, size=bits.size, dtype=np.uint32) << 31)
    q = bits.view(np.float32)
    assert np.array_equal(oracle.encode(q, fmt), nearest_code(q, name))


def test_signed_zero_and_underflow():
    q = np.array([0.0, -0.0, -1e-30, 1e-30, -2.0 ** -11], np.float32)
    assert list(oracle.encode(q, oracle.FMT_E4M3)) == [0, 0x80, 0x80, 0, 0x80]
    assert list(oracle.encode(q, oracle.FMT_E2M1)) == [0, 0x8, 0x8, 0, 0x8]


def test_saturation():
    q = np.array([448, 449, 464, 1e6, -500, 6, 7, -100], np.float32)
    e4 = oracle.encode(q[:5], oracle.FMT_E4M3)
    assert list(e4) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    e2 = oracle.encode(q[5:], oracle.FMT_E2M1)
    assert list(e2) == [0x7, 0x7, 0xF]


@pytest.mark.parametrize("name,fmt", FMTS)
def test_decode_roundtrip(name, fmt):
    """Encoding each representable value returns its own code."""
    t = decode_table(name)
    vals = np.concatenate([t, -t[1:]]).astype(np.float32)
    codes = oracle.encode(vals, fmt)
    assert np.array_equal(decode(codes, name), vals.astype(np.float64))
