"""Pins of the oracle's whole cast (CPU only): worked examples, invariants,
layouts and packing, and an exact-arithmetic brute force on tiny inputs."""
import os

import numpy as np
import pytest

import oracle
from bruteforce import (F32_1E4, FMT_MAX, cast_bruteforce, decode,
                        decode_table)
from precision_quantization_token_gb300.inputs import (bf16_bits_to_f32,
                                                       f32_to_bf16_bits,
                                                       random_bf16)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MODES = {"fp32": oracle.SCALE_FP32, "pow2": oracle.SCALE_FP32_POW2,
         "ue8m0": oracle.SCALE_UE8M0}
FMTS = {"e4m3": oracle.FMT_E4M3, "e2m1": oracle.FMT_E2M1}


def read_worked_row(fname):
    xs, codes = [], []
    for line in open(os.path.join(GOLDEN, fname)):
        if line.startswith("#") or not line.strip():
            continue
        x, c = line.split()[:2]
        xs.append(float(x))
        codes.append(int(c, 16))
    return np.array(xs, np.float32), np.array(codes)


def unpack_e2m1(packed):
    packed = np.asarray(packed, np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


@pytest.mark.parametrize("mode", ["fp32", "pow2", "ue8m0"])
def test_worked_row_e4m3(mode):
    x, want = read_worked_row("e4m3_unit_scale_row.txt")
    bits = f32_to_bf16_bits(x)[None, :]
    assert np.array_equal(bf16_bits_to_f32(bits)[0], x)   # exact BF16 values
    codes, scales = oracle.per_token_cast(bits, 16, 16, oracle.FMT_E4M3,
                                          MODES[mode], oracle.LAYOUT_ROW_MAJOR)
    assert list(codes[0]) == list(want)
    if mode == "ue8m0":
        assert scales.view(np.uint8)[0, 0] == 127
    else:
        assert scales[0, 0] == 1.0


def test_worked_row_e2m1():
    x, want = read_worked_row("e2m1_unit_scale_row.txt")
    bits = f32_to_bf16_bits(x)[None, :]
    codes, scales = oracle.per_token_cast(bits, 16, 16, oracle.FMT_E2M1,
                                          oracle.SCALE_UE8M0,
                                          oracle.LAYOUT_ROW_MAJOR)
    assert list(unpack_e2m1(codes)[0]) == list(want)
    assert list(codes[0]) == [0x07, 0x22, 0x44, 0x66, 0x8F, 0x80, 0x21, 0x56]
    assert scales.view(np.uint8)[0, 0] == 127


def _amax_rows(fmt_name, group):
    """One row per positive BF16 value a >= 1e-4 whose amax is a (at a
    seeded position) with smaller seeded entries of both signs."""
    bits = np.arange(0x3800, 0x7F80, dtype=np.uint32)
    a = (bits << 16).view(np.float32)
    a = a[a >= F32_1E4]
    rng = np.random.default_rng(7)
    frac = rng.uniform(-1, 1, size=(a.size, group)).astype(np.float32)
    rows = f32_to_bf16_bits(frac * a[:, None])
    mag = bf16_bits_to_f32(rows)
    rows[np.abs(mag) > a[:, None]] = 0          # keep |x| <= a after rounding
    pos = rng.integers(0, group, size=a.size)
    rows[np.arange(a.size), pos] = f32_to_bf16_bits(a)
    return rows, pos


@pytest.mark.parametrize("fmt_name", ["e4m3", "e2m1"])
def test_fp32_mode_amax_element_hits_format_max(fmt_name):
    """Non-power-of-two scale: the amax element's code is +-fmt_max."""
    group = 16
    rows, pos = _amax_rows(fmt_name, group)
    codes, _ = oracle.per_token_cast(rows, group, group, FMTS[fmt_name],
                                     oracle.SCALE_FP32, oracle.LAYOUT_ROW_MAJOR)
    if fmt_name == "e2m1":
        codes = unpack_e2m1(codes)
    top = decode(codes[np.arange(rows.shape[0]), pos], fmt_name)
    assert np.all(np.abs(top) == FMT_MAX[fmt_name])


@pytest.mark.parametrize("fmt_name", ["e4m3", "e2m1"])
def test_pow2_mode_amax_element_in_top_binade(fmt_name):
    """Power-of-two scale: fmt_max/2 <= |code(amax)| <= fmt_max."""
    group = 16
    rows, pos = _amax_rows(fmt_name, group)
    codes, _ = oracle.per_token_cast(rows, group, group, FMTS[fmt_name],
                                     oracle.SCALE_UE8M0,
                                     oracle.LAYOUT_ROW_MAJOR)
    if fmt_name == "e2m1":
        codes = unpack_e2m1(codes)
    top = np.abs(decode(codes[np.arange(rows.shape[0]), pos], fmt_name))
    assert np.all(top <= FMT_MAX[fmt_name])
    assert np.all(top >= FMT_MAX[fmt_name] / 2)


def _scales_as_float(scales, mode, M, G, layout):
    if mode == "ue8m0":
        b = scales.view(np.uint8)
        if layout == "row":
            e = b.reshape(M, -1)[:, :G]
        else:
            e = np.stack([b.reshape(scales.shape[0], -1, 4)[j // 4, :M, j % 4]
                          for j in range(G)], axis=1)
        return np.ldexp(1.0, e.astype(np.int64) - 127)
    s = scales.astype(np.float64)
    return s[:M, :G] if layout == "row" else s[:G, :M].T


@pytest.mark.parametrize("fmt_name", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "pow2", "ue8m0"])
@pytest.mark.parametrize("group", [16, 32, 64, 128])
def test_dequantisation_error_bound(fmt_name, mode, group):
    """|x - dec(code)*s| <= (gap/2)*s + |x|*2^-23 for every element, where
    gap is the distance from dec(code) to its neighbour on x's side."""
    M, K = 37, 256
    bits = random_bf16(100 + group, M, K, scale=3.0)
    bits[3] = 0                                         # all-zero row
    bits[5, :group] = np.uint16(0x0005)                 # denormal group
    codes, scales = oracle.per_token_cast(bits, K, group, FMTS[fmt_name],
                                          MODES[mode], oracle.LAYOUT_ROW_MAJOR)
    if fmt_name == "e2m1":
        codes = unpack_e2m1(codes)
    x = bf16_bits_to_f32(bits).astype(np.float64)
    s = np.repeat(_scales_as_float(scales, mode, M, K // group, "row"),
                  group, axis=1)
    d = decode(codes, fmt_name)
    table = decode_table(fmt_name)
    mag = np.abs(d)
    idx = np.searchsorted(table, mag)
    q = x / s
    toward_up = np.abs(q) > mag
    up = table[np.clip(idx + 1, 0, table.size - 1)] - mag
    dn = mag - table[np.clip(idx - 1, 0, table.size - 1)]
    gap = np.where(toward_up, up, dn)
    gap = np.where(gap == 0, table[-1] - table[-2], gap)
    err = np.abs(x - d * s)
    bound = 0.5 * gap * s + np.abs(x) * 2.0 ** -23
    assert np.all(err <= bound)
    # the sign always follows x (zeros keep theirs)
    assert np.all(np.signbit(d) == np.signbit(x))


@pytest.mark.parametrize("fmt_name", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "pow2", "ue8m0"])
def test_bruteforce_tiny(fmt_name, mode):
    """Exact-arithmetic cast of tiny random rows equals the oracle."""
    for seed, (M, K, group) in enumerate([(3, 32, 16), (2, 128, 32),
                                          (1, 128, 128), (2, 128, 64)]):
        bits = random_bf16(500 + seed, M, K, scale=10.0 ** (seed - 2))
        if seed == 0:
            bits[1, :16] = 0x8000                         # a -0 group
            bits[2, 16:] = np.uint16(0x0003)              # denormal group
        codes, scales = oracle.per_token_cast(bits, K, group, FMTS[fmt_name],
                                              MODES[mode],
                                              oracle.LAYOUT_ROW_MAJOR)
        if fmt_name == "e2m1":
            codes = unpack_e2m1(codes)
        x = bf16_bits_to_f32(bits)
        for m in range(M):
            want_codes, want_scales = cast_bruteforce(x[m].tolist(), group,
                                                      fmt_name, mode)
            assert list(codes[m]) == want_codes
            if mode == "ue8m0":
                got = list(scales.view(np.uint8)[m, :K // group])
            else:
                got = scales[m, :K // group].tolist()
            assert got == want_scales


def test_ue8m0_packing_order_and_pad_bytes():
    """Group 4w+b lands in byte b of int32 word w; the unused bytes of a
    partly filled last word are zero; entries past it are untouched."""
    G, group = 6, 16
    amax = 448.0 * 2.0 ** np.arange(G)                   # byte 127 + j
    x = np.zeros((2, G * group), np.float32)
    x[:, ::group] = amax
    bits = f32_to_bf16_bits(x)
    scales = np.full((2, 3), -1, np.int32)               # 2 words + 1 spare
    codes, scales = oracle.per_token_cast(bits, G * group, group,
                                          oracle.FMT_E4M3, oracle.SCALE_UE8M0,
                                          oracle.LAYOUT_ROW_MAJOR,
                                          scales=scales)
    b = scales.view(np.uint8).reshape(2, 12)
    assert list(b[0, :8]) == [127, 128, 129, 130, 131, 132, 0, 0]
    assert list(b[0, 8:]) == [0xFF] * 4
    assert scales.view(np.uint32)[0, 0] == 127 | 128 << 8 | 129 << 16 | 130 << 24


@pytest.mark.parametrize("mode", ["fp32", "pow2", "ue8m0"])
@pytest.mark.parametrize("M", [1, 3, 5, 254])
def test_transposed_layout_matches_row_major(mode, M):
    """DeepGEMM-style layout: [G or ceil(G/4)][M_pad], M_pad = ceil(M/4)*4;
    the same values as the row-major layout, pad columns left untouched."""
    K, group = 320, 32
    G = K // group
    bits = random_bf16(900 + M, M, K)
    c_row, s_row = oracle.per_token_cast(bits, K, group, oracle.FMT_E4M3,
                                         MODES[mode], oracle.LAYOUT_ROW_MAJOR)
    r, c, dt = oracle.scale_shape(M, K, group, MODES[mode],
                                  oracle.LAYOUT_TRANSPOSED)
    assert c == (M + 3) // 4 * 4
    sent = np.full((r, c), -7, dt)
    c_t, s_t = oracle.per_token_cast(bits, K, group, oracle.FMT_E4M3,
                                     MODES[mode], oracle.LAYOUT_TRANSPOSED,
                                     scales=sent)
    assert np.array_equal(c_row, c_t)
    assert np.array_equal(_scales_as_float(s_row, mode, M, G, "row"),
                          _scales_as_float(s_t, mode, M, G, "transposed"))
    assert np.all(s_t[:, M:] == -7)


def test_input_row_stride_and_code_nibble_order():
    K = 32
    x = np.zeros((2, 48), np.float32)
    x[:, K:] = 1e30                        # stride padding must be ignored
    x[0, 0], x[1, 1] = 6.0, 6.0
    bits = f32_to_bf16_bits(x)
    codes, _ = oracle.per_token_cast(bits, K, 16, oracle.FMT_E2M1,
                                     oracle.SCALE_UE8M0,
                                     oracle.LAYOUT_ROW_MAJOR)
    assert codes[0, 0] == 0x07 and codes[1, 0] == 0x70


def test_nonfinite_input_is_rejected():
    bits = np.zeros((1, 16), np.uint16)
    bits[0, 3] = 0x7FC0                    # NaN
    with pytest.raises(ValueError):
        oracle.per_token_cast(bits, 16, 16, oracle.FMT_E4M3,
                              oracle.SCALE_FP32, oracle.LAYOUT_ROW_MAJOR)


def test_threaded_split_is_identical():
    bits = random_bf16(77, 64, 512)
    a = oracle.per_token_cast(bits, 512, 64, oracle.FMT_E4M3,
                              oracle.SCALE_FP32, oracle.LAYOUT_TRANSPOSED)
    b = oracle.per_token_cast(bits, 512, 64, oracle.FMT_E4M3,
                              oracle.SCALE_FP32, oracle.LAYOUT_TRANSPOSED,
                              threads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
