"""Pins of the oracle's fused SwiGLU + cast (CPU only).

The oracle forms y = gate * up / (1 + e^-gate) in double and rounds it once
to fp32.  Here y is evaluated with 60-digit mpmath arithmetic and rounded to
fp32 exactly (tests/bruteforce.rn_f32), and the cast of the product row is
redone with exact rationals.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bruteforce import cast_bruteforce, rn_f32
from precision_quantization_token_gb300.inputs import (bf16_bits_to_f32,
                                                       random_bf16)

mpmath = pytest.importorskip("mpmath")
mpmath.mp.dps = 60


def exact_swiglu_f32(g: float, u: float) -> float:
    g_, u_ = mpmath.mpf(g), mpmath.mpf(u)
    y = g_ * u_ / (1 + mpmath.exp(-g_))
    if y == 0:
        return 0.0 if (g * u >= 0 and not np.signbit(g * u)) else -0.0
    sign, man, exp, _ = y._mpf_
    f = Fraction(int(man)) * Fraction(2) ** int(exp)
    return rn_f32(-f if sign else f)


def f32_ulp_distance(a: float, b: float) -> int:
    ia = np.array([a], np.float32).view(np.int32)[0]
    ib = np.array([b], np.float32).view(np.int32)[0]
    ia = ia if ia >= 0 else -(ia & 0x7FFFFFFF)
    ib = ib if ib >= 0 else -(ib & 0x7FFFFFFF)
    return abs(int(ia) - int(ib))


def test_swiglu_value_matches_high_precision():
    rng = np.random.default_rng(3)
    pts = [(0.0, 1.0), (1.0, 1.0), (-1.0, 1.0), (20.0, -3.0), (-20.0, 2.0),
           (-88.0, 1.0), (-100.0, 1e30), (1e-30, 1.0), (-1e-30, -1.0),
           (3.5, 0.0), (0.6931471805599453, 1.0)]
    g = rng.standard_normal(2000).astype(np.float32) * 4
    u = rng.standard_normal(2000).astype(np.float32) * 2
    pts += list(zip(g.tolist(), u.tolist()))
    exact = 0
    for gi, ui in pts:
        got = oracle.swiglu_value(gi, ui)
        want = exact_swiglu_f32(gi, ui)
        d = f32_ulp_distance(got, want)
        assert d <= 1, (gi, ui, got, want)
        exact += d == 0
    assert exact >= 0.999 * len(pts)


def test_silu_closed_forms():
    # silu(0) = 0; silu(ln 3) = (3/4) ln 3; silu(-v) = silu(v) - v.
    assert oracle.swiglu_value(0.0, 5.0) == 0.0
    ln3 = float(np.float32(np.log(3.0)))
    want = exact_swiglu_f32(ln3, 1.0)
    assert oracle.swiglu_value(ln3, 1.0) == want
    assert abs(want - 0.75 * ln3) < 1e-6
    for v in [0.5, 1.0, 2.0, 7.0]:
        assert abs(oracle.swiglu_value(-v, 1.0) -
                   (oracle.swiglu_value(v, 1.0) - v)) < 4e-7 * max(1, v)


@pytest.mark.parametrize("mode", ["fp32", "pow2", "ue8m0"])
@pytest.mark.parametrize("fmt_name", ["e4m3", "e2m1"])
def test_bruteforce_tiny_swiglu(mode, fmt_name):
    fmt = oracle.FMT_E4M3 if fmt_name == "e4m3" else oracle.FMT_E2M1
    mode_id = {"fp32": oracle.SCALE_FP32, "pow2": oracle.SCALE_FP32_POW2,
               "ue8m0": oracle.SCALE_UE8M0}[mode]
    M, N, group = 3, 64, 32
    bits = random_bf16(41, M, 2 * N, scale=2.0)
    bits[1, :N] = 0                                   # gate 0 -> y = 0
    codes, scales = oracle.swiglu_per_token_cast(bits, N, group, fmt, mode_id,
                                                 oracle.LAYOUT_ROW_MAJOR)
    if fmt_name == "e2m1":
        unpacked = np.empty((M, N), np.uint8)
        unpacked[:, 0::2], unpacked[:, 1::2] = codes & 0xF, codes >> 4
        codes = unpacked
    x = bf16_bits_to_f32(bits)
    for m in range(M):
        y = [exact_swiglu_f32(float(x[m, k]), float(x[m, N + k]))
             for k in range(N)]
        want_codes, want_scales = cast_bruteforce(y, group, fmt_name, mode)
        assert list(codes[m]) == want_codes
        got = (list(scales.view(np.uint8)[m, :N // group]) if mode == "ue8m0"
               else scales[m, :N // group].tolist())
        assert got == want_scales


def test_gate_is_first_half():
    """With up = 1 everywhere, the codes are those of silu(gate) alone; with
    the halves swapped they are not."""
    N, group = 32, 32
    g = np.linspace(-4, 4, N, dtype=np.float32)
    from precision_quantization_token_gb300.inputs import f32_to_bf16_bits
    row = np.concatenate([g, np.ones(N, np.float32)])[None, :]
    bits = f32_to_bf16_bits(row)
    codes, _ = oracle.swiglu_per_token_cast(bits, N, group, oracle.FMT_E4M3,
                                            oracle.SCALE_FP32,
                                            oracle.LAYOUT_ROW_MAJOR)
    gf = bf16_bits_to_f32(bits[0, :N])
    y = [exact_swiglu_f32(float(v), 1.0) for v in gf]
    want, _ = cast_bruteforce(y, group, "e4m3", "fp32")
    assert list(codes[0]) == want
    swapped = np.concatenate([bits[:, N:], bits[:, :N]], axis=1)
    codes2, _ = oracle.swiglu_per_token_cast(swapped, N, group,
                                             oracle.FMT_E4M3,
                                             oracle.SCALE_FP32,
                                             oracle.LAYOUT_ROW_MAJOR)
    assert list(codes2[0]) != want
