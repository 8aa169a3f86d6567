"""Pins of the oracle's dequantization and cast-and-cast-back (CPU only).

Dequantization: code value (OCP definitions) times the group scale in one
IEEE fp32 multiply, then (for BF16 output) round to nearest even.  Checked
against the value-space decode table of tests/bruteforce.py and an
independent numpy BF16 rounding; cast-back against dequant(cast(x)) and the
quantisation error bound.
"""
import numpy as np
import pytest

import oracle
from bruteforce import FMT_MAX, decode, decode_table
from precision_quantization_token_gb300.inputs import (bf16_bits_to_f32,
                                                       f32_to_bf16_bits,
                                                       random_bf16)

FMTS = {"e4m3": oracle.FMT_E4M3, "e2m1": oracle.FMT_E2M1}
MODES = {"fp32": oracle.SCALE_FP32, "pow2": oracle.SCALE_FP32_POW2,
         "ue8m0": oracle.SCALE_UE8M0}


def _all_codes(fmt):
    if fmt == "e4m3":
        c = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
        return c, c.copy()
    nib = np.arange(16, dtype=np.uint8)
    packed = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    return packed, nib


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_decode_every_code_with_unit_scale(fmt):
    stored, unpacked = _all_codes(fmt)
    K = unpacked.size
    K16 = -(-K // 16) * 16
    codes = np.zeros((1, K16 if fmt == "e4m3" else K16 // 2), np.uint8)
    codes[0, :stored.size] = stored
    scales = np.ones((1, K16 // 16), np.float32)
    y = oracle.per_token_dequant(codes, scales, K16, 16, FMTS[fmt],
                                 oracle.SCALE_FP32, oracle.LAYOUT_ROW_MAJOR,
                                 out_fp32=True)
    got = y[0, :K].astype(np.float64)
    want = decode(unpacked, fmt)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "ue8m0"])
@pytest.mark.parametrize("layout", ["row", "transposed"])
def test_dequant_is_one_fp32_multiply_then_bf16_rne(fmt, mode, layout):
    M, K, group = 9, 256, 32
    rng = np.random.default_rng(3)
    nbytes = K if fmt == "e4m3" else K // 2
    codes = rng.integers(0, 256, size=(M, nbytes), dtype=np.uint8)
    if fmt == "e4m3":
        codes[(codes & 0x7F) == 0x7F] = 0x12          # no NaN codes
    G = K // group
    lay = oracle.LAYOUT_ROW_MAJOR if layout == "row" else oracle.LAYOUT_TRANSPOSED
    if mode == "ue8m0":
        words = (G + 3) // 4
        b = rng.integers(100, 150, size=(M, words * 4), dtype=np.uint8)
        s_val = np.ldexp(1.0, b[:, :G].astype(np.int64) - 127)
        scales = b.view(np.int32) if layout == "row" else np.ascontiguousarray(
            b.reshape(M, words, 4).transpose(1, 0, 2)).reshape(words, M * 4).view(np.int32)
    else:
        s_val = rng.uniform(1e-3, 10, size=(M, G)).astype(np.float32)
        scales = s_val if layout == "row" else np.ascontiguousarray(s_val.T)
    y32 = oracle.per_token_dequant(codes, scales, K, group, FMTS[fmt],
                                   MODES[mode], lay, out_fp32=True)
    y16 = oracle.per_token_dequant(codes, scales, K, group, FMTS[fmt],
                                   MODES[mode], lay)
    if fmt == "e4m3":
        unpacked = codes
    else:
        unpacked = np.empty((M, K), np.uint8)
        unpacked[:, 0::2], unpacked[:, 1::2] = codes & 0xF, codes >> 4
    dec = decode(unpacked, fmt).astype(np.float32)
    s_rep = np.repeat(np.asarray(s_val, np.float32), group, axis=1)
    want32 = dec * s_rep                                  # numpy fp32 IEEE
    assert np.array_equal(y32.view(np.uint32), want32.view(np.uint32))
    assert np.array_equal(y16, f32_to_bf16_bits(want32))


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "pow2", "ue8m0"])
@pytest.mark.parametrize("group", [16, 128])
def test_cast_back_equals_dequant_of_cast(fmt, mode, group):
    M, K = 21, 512
    bits = random_bf16(7 + group, M, K, scale=4.0)
    bits[2] = 0x8000                                    # a -0 row
    bits[3, :group] = np.uint16(0x0007)                 # a denormal group
    back = oracle.per_token_cast_back(bits, K, group, FMTS[fmt], MODES[mode],
                                      threads=3)
    codes, scales = oracle.per_token_cast(bits, K, group, FMTS[fmt],
                                          MODES[mode],
                                          oracle.LAYOUT_ROW_MAJOR)
    deq = oracle.per_token_dequant(codes, scales, K, group, FMTS[fmt],
                                   MODES[mode], oracle.LAYOUT_ROW_MAJOR)
    assert np.array_equal(back, deq)
    # quantisation error bound: half the code gap times the scale, plus the
    # fp32 quotient and BF16 roundings
    x = bf16_bits_to_f32(bits).astype(np.float64)
    xb = bf16_bits_to_f32(back).astype(np.float64)
    if mode == "ue8m0":
        e = scales.view(np.uint8).reshape(M, -1)[:, :K // group]
        s = np.ldexp(1.0, e.astype(np.int64) - 127)
    else:
        s = scales[:, :K // group].astype(np.float64)
    s = np.repeat(s, group, axis=1)
    table = decode_table(fmt)
    max_gap = np.max(np.diff(table))
    bound = (0.5 * max_gap * s + np.abs(x) * 2.0 ** -23
             + np.abs(xb) * 2.0 ** -8)
    assert np.all(np.abs(x - xb) <= bound)
    assert np.all(np.signbit(xb) == np.signbit(x))
    assert np.all(np.abs(xb) <= FMT_MAX[fmt] * s * (1 + 2.0 ** -8))


def test_bf16_rounding_ties_and_neighbours():
    """Code 1.0 (E4M3 0x38) times fp32 scales whose low 16 bits are exactly
    half a BF16 ulp (ties, both even and odd upper halves) or one unit either
    side: the BF16 output must be the nearest, ties to even."""
    uppers = np.array([0x3F80, 0x3F81, 0x4000, 0x4001, 0x3C7F, 0x3C80,
                       0x007F, 0x0080, 0x7F7E], np.uint32)
    lows = np.array([0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF], np.uint32)
    s_bits = (uppers[:, None] << 16 | lows[None, :]).reshape(-1)
    n = -(-s_bits.size // 1) * 1
    K = 16 * n
    codes = np.full((1, K), 0x38, np.uint8)
    scales = s_bits.view(np.float32)[None, :]
    y = oracle.per_token_dequant(codes, scales, K, 16, oracle.FMT_E4M3,
                                 oracle.SCALE_FP32, oracle.LAYOUT_ROW_MAJOR)
    want = f32_to_bf16_bits(s_bits.view(np.float32))
    assert np.array_equal(y[0, ::16], want)
    # the tie cases themselves round to the even upper half
    ties = y[0, ::16].reshape(len(uppers), len(lows))[:, 0]
    assert np.all(ties % 2 == 0)
