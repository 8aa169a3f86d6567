"""Pins of the oracle's RMSNorm and its fused per-token cast (CPU only).

RMSNorm follows its published definition (Zhang and Sennrich, "Root Mean
Square Layer Normalization", 2019): y_k = w_k x_k / sqrt(eps + mean_j x_j^2),
formed in double and rounded once to fp32.  Pins: hand-worked values
(tests/golden/rmsnorm_small.txt), exact invariances (power-of-two scaling of
x with eps = 0, power-of-two gain, channel permutation), the unit RMS of the
output, and -- for the fused cast -- equality with the separately pinned
per-token cast on rows whose output is exactly representable in BF16.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rmsnorm_small.txt")


def bf16(values):
    a = np.asarray(values, np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)   # exact for these values


def random_rows(M, K, seed, spread=True):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((M, K)).astype(np.float32)
    if spread:
        v *= np.exp2(rng.integers(-10, 11, (M, 1))).astype(np.float32)
    return bf16(v)


def _vals(field, K, fill):
    if field.startswith("*"):
        return [float(field[1:])] * K
    vals = [float(t) for t in field.split(";")]
    return vals + [fill] * (K - len(vals))


def golden_cases():
    out = []
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        K, eps, xs, ws, ys = line.split()
        K = int(K)
        want = [int(t, 16) for t in ys.split(";")]
        out.append((K, float(eps), _vals(xs, K, 0.0), _vals(ws, K, 1.0), want))
    return out


@pytest.mark.parametrize("K,eps,x,w,want", golden_cases())
def test_golden(K, eps, x, w, want):
    y = oracle.rmsnorm_values(bf16([x]), bf16(w), K, eps)
    got = y[0, :len(want)].view(np.uint32).tolist()
    assert got == want, [hex(g) for g in got]


@pytest.mark.parametrize("k", [-40, -7, 3, 25])
def test_power_of_two_scaling_of_x_changes_nothing(k):
    """eps = 0: x -> 2^k x scales every square by 4^k and the root by 2^k."""
    x = random_rows(8, 256, seed=k + 100, spread=False)
    w = random_rows(1, 256, seed=7)[0]
    xs = bf16(((x.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** k)))
    a = oracle.rmsnorm_values(x, w, 256, 0.0)
    b = oracle.rmsnorm_values(xs, w, 256, 0.0)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_power_of_two_gain_scales_the_output():
    x = random_rows(8, 128, seed=1)
    w = random_rows(1, 128, seed=2)[0]
    w4 = bf16(((w.astype(np.uint32) << 16).view(np.float32) * np.float32(4.0)))
    a = oracle.rmsnorm_values(x, w, 128, 1e-6)
    b = oracle.rmsnorm_values(x, w4, 128, 1e-6)
    assert np.array_equal(a * np.float32(4.0), b)


def test_channel_permutation_permutes_the_output():
    x = random_rows(6, 160, seed=3)
    w = random_rows(1, 160, seed=4)[0]
    perm = np.random.default_rng(5).permutation(160)
    a = oracle.rmsnorm_values(x, w, 160, 1e-5)
    b = oracle.rmsnorm_values(np.ascontiguousarray(x[:, perm]), w[perm], 160, 1e-5)
    assert np.array_equal(a[:, perm], b)


def test_unit_gain_output_has_unit_rms():
    """w = 1, eps = 0: mean(y^2) = 1 up to the fp32 rounding of each y."""
    x = random_rows(16, 1024, seed=6)
    w = bf16(np.ones(1024))
    y = oracle.rmsnorm_values(x, w, 1024, 0.0).astype(np.float64)
    ms = (y * y).mean(axis=1)
    assert np.all(np.abs(ms - 1.0) <= 2.0 ** -22)


def test_eps_shrinks_the_output():
    x = random_rows(4, 64, seed=8, spread=False)
    w = random_rows(1, 64, seed=9)[0]
    a = np.abs(oracle.rmsnorm_values(x, w, 64, 0.0))
    b = np.abs(oracle.rmsnorm_values(x, w, 64, 0.5))
    assert np.all(b <= a) and np.all(b[a > 0] < a[a > 0])


FMTS = [oracle.FMT_E4M3, oracle.FMT_E2M1]
MODES = [oracle.SCALE_FP32, oracle.SCALE_FP32_POW2, oracle.SCALE_UE8M0]
LAYOUTS = [oracle.LAYOUT_ROW_MAJOR, oracle.LAYOUT_TRANSPOSED]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_fused_cast_is_the_per_token_cast_of_y(fmt, mode, layout):
    """x = +-c per row (rms = c, eps = 0) makes y = +-w exactly, a BF16 row:
    the fused cast must equal the per-token cast of that row."""
    M, K, group = 12, 256, 32
    rng = np.random.default_rng(10)
    c = np.exp2(rng.integers(-5, 6, (M, 1))).astype(np.float32)
    sign = np.where(rng.random((M, K)) < 0.5, -1.0, 1.0).astype(np.float32)
    x = bf16(c * sign)
    w = random_rows(1, K, seed=11)[0]
    y_bits = bf16((sign * (w.astype(np.uint32) << 16).view(np.float32)))
    got = oracle.rmsnorm_per_token_cast(x, w, K, 0.0, group, fmt, mode, layout)
    want = oracle.per_token_cast(y_bits, K, group, fmt, mode, layout)
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1].view(np.uint32), want[1].view(np.uint32))


def test_zero_row():
    """eps > 0: a zero row gives y = 0, all-zero codes and the floor scale;
    eps = 0: 0/0, reported as outside the op's domain."""
    x = np.zeros((2, 128), np.uint16)
    w = random_rows(1, 128, seed=12)[0]
    codes, scales = oracle.rmsnorm_per_token_cast(x, w, 128, 1e-6, 128,
                                                  oracle.FMT_E4M3,
                                                  oracle.SCALE_FP32,
                                                  oracle.LAYOUT_ROW_MAJOR)
    assert not (codes & 0x7F).any()           # +-0: the sign of w * 0 is kept
    assert np.array_equal(codes[0] >> 7, (w >> 15).astype(np.uint8))
    assert np.all(scales == np.float32(np.float32(1e-4) / np.float32(448)))
    with pytest.raises(ValueError):
        oracle.rmsnorm_per_token_cast(x, w, 128, 0.0, 128, oracle.FMT_E4M3,
                                      oracle.SCALE_FP32, oracle.LAYOUT_ROW_MAJOR)
