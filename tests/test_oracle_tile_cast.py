"""Pins of the oracle's per-block and per-channel casts (CPU only).

The per-block cast shares one scale across a square block of rows x
channels; the per-channel cast shares one across a whole column.  These
tests pin the oracle against:

* a brute force written from the op's definition with numpy and the
  value-space references in tests/bruteforce.py (block / column amax by
  numpy, the scale with exact rationals, codes by nearest-value search of
  the IEEE fp32 quotient);
* reductions to the per-token cast, which has its own pins: a one-row
  per-block cast is a per-token cast with group = block, and a per-channel
  cast of an M-row matrix (M a legal group size) is the transposed
  per-token cast of the transposed matrix with group = M;
* symmetry (square blocks: casting x^T gives the transposed result),
  special blocks, and the padding and untouched-memory rules.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bruteforce import FMT_MAX, decode, nearest_code, rn_f32, scale_bruteforce

FMTS = [("e4m3", oracle.FMT_E4M3), ("e2m1", oracle.FMT_E2M1)]
MODES = [("fp32", oracle.SCALE_FP32), ("pow2", oracle.SCALE_FP32_POW2),
         ("ue8m0", oracle.SCALE_UE8M0)]


def bf16_matrix(M, K, seed):
    """Normal values with per-row and per-column spread, exact zeros, -0,
    BF16 denormals and a few outliers: every block / column amax differs."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 7, (M, 1)))
    v = v * np.exp2(rng.integers(-4, 5, (1, K)))
    v[rng.random((M, K)) < 0.02] = 0.0
    v[rng.random((M, K)) < 0.02] = -0.0
    bits = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    den = rng.random((M, K)) < 0.01
    bits[den] = (rng.integers(1, 128, den.sum()) |
                 (rng.integers(0, 2, den.sum()) << 15)).astype(np.uint16)
    out = rng.random((M, K)) < 0.002
    bits[out] = (np.float32(300.0).view(np.uint32) >> 16).astype(np.uint16)
    return bits


def as_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def unpack(codes, fmt):
    if fmt == "e4m3":
        return codes
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = codes & 0xF
    out[..., 1::2] = codes >> 4
    return out


def scale_entries(scales, n, mode):
    """The first n entries of a scale row / vector: floats, or UE8M0 bytes."""
    if mode == "ue8m0":
        return scales.view(np.uint8).reshape(-1)[:n].astype(np.int64)
    return scales.view(np.float32).reshape(-1)[:n]


def brute_group(vals, fmt, mode):
    """Codes and scale of one scale group given as fp32 values (numpy fp32
    division is the IEEE quotient the op prescribes)."""
    amax = float(np.abs(vals.astype(np.float64)).max()) if vals.size else 0.0
    s, e = scale_bruteforce(amax, fmt, mode)
    q = vals.astype(np.float32) / np.float32(s)
    return nearest_code(q, fmt), (e if mode == "ue8m0" else s)


# ------------------------------------------------------------- brute force

@pytest.mark.parametrize("fname,fmt", FMTS)
@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("M,K,block", [(37, 48, 16), (5, 64, 32),
                                       (130, 256, 128), (64, 96, 64)])
def test_per_block_bruteforce(fname, fmt, mname, mode, M, K, block):
    bits = bf16_matrix(M, K, seed=M * 1000 + K + block)
    codes, scales = oracle.per_block_cast(bits, K, block, fmt, mode)
    got = unpack(codes, fname)
    x = as_f32(bits)
    nc = -(-K // block)
    for rb in range(-(-M // block)):
        srow = scale_entries(scales[rb], nc, mname)
        for cb in range(nc):
            blk = x[rb * block:(rb + 1) * block, cb * block:(cb + 1) * block]
            want, s = brute_group(blk, fname, mname)
            assert srow[cb] == s, (rb, cb, srow[cb], s)
            have = got[rb * block:(rb + 1) * block, cb * block:(cb + 1) * block]
            assert np.array_equal(have, want), (rb, cb)


@pytest.mark.parametrize("fname,fmt", FMTS)
@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("M,K", [(37, 48), (3, 16), (200, 40), (1, 8)])
def test_per_channel_bruteforce(fname, fmt, mname, mode, M, K):
    bits = bf16_matrix(M, K, seed=7 * M + K)
    codes, scales = oracle.per_channel_cast(bits, K, fmt, mode, threads=3)
    got = unpack(codes, fname)
    x = as_f32(bits)
    sv = scale_entries(scales, K, mname)
    for k in range(K):
        want, s = brute_group(x[:, k], fname, mname)
        assert sv[k] == s, (k, sv[k], s)
        assert np.array_equal(got[:, k], want), k


def test_per_block_tiny_exact():
    """A 2x2 matrix in one 16-block, every step with exact rationals: amax
    3.5 -> s = RN(3.5/448) = 2^-7 exactly; codes of x * 128."""
    bits = np.zeros((2, 16), np.uint16)
    vals = [[3.5, -1.25], [0.0078125, -0.0]]
    for r in range(2):
        for c in range(2):
            bits[r, c] = np.float32(vals[r][c]).view(np.uint32) >> 16
    codes, scales = oracle.per_block_cast(bits, 16, 16, oracle.FMT_E4M3,
                                          oracle.SCALE_FP32)
    assert scales[0, 0] == rn_f32(Fraction(7, 2) / 448) == 2.0 ** -7
    assert list(decode(codes[0, :2], "e4m3")) == [448.0, -160.0]
    assert list(decode(codes[1, :2], "e4m3")) == [1.0, 0.0]
    assert codes[1, 1] == 0x80          # -0 keeps its sign
    assert not codes[:, 2:].any()


# ------------------------------------------------- reductions to per-token

@pytest.mark.parametrize("fname,fmt", FMTS)
@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("block", [16, 32, 64, 128])
def test_one_row_per_block_is_per_token(fname, fmt, mname, mode, block):
    K = 4 * block + block            # 5 blocks: a partly filled UE8M0 word
    bits = bf16_matrix(1, K, seed=block)
    c_b, s_b = oracle.per_block_cast(bits, K, block, fmt, mode)
    c_t, s_t = oracle.per_token_cast(bits, K, block, fmt, mode,
                                     oracle.LAYOUT_ROW_MAJOR)
    assert np.array_equal(c_b, c_t)
    assert np.array_equal(s_b.view(np.uint32), s_t.view(np.uint32))


@pytest.mark.parametrize("fname,fmt", FMTS)
@pytest.mark.parametrize("mname,mode", MODES)
@pytest.mark.parametrize("M", [16, 32, 64, 128])
def test_per_channel_is_transposed_per_token(fname, fmt, mname, mode, M):
    K = 40
    bits = bf16_matrix(M, K, seed=M + 5)
    c_c, s_c = oracle.per_channel_cast(bits, K, fmt, mode)
    xt = np.ascontiguousarray(bits.T)                  # [K, M]
    c_t, s_t = oracle.per_token_cast(xt, M, M, fmt, mode,
                                     oracle.LAYOUT_ROW_MAJOR)
    assert np.array_equal(unpack(c_c, fname), unpack(c_t, fname).T)
    # per-token: one group per row -> word 0 of row k (UE8M0: byte 0)
    if mname == "ue8m0":
        assert np.array_equal(scale_entries(s_c, K, mname),
                              s_t.view(np.uint8)[:, 0].astype(np.int64))
    else:
        assert np.array_equal(s_c.view(np.uint32), s_t[:, 0].view(np.uint32))


# ------------------------------------------------ symmetry, special cases

@pytest.mark.parametrize("mname,mode", MODES)
def test_square_blocks_commute_with_transpose(mname, mode):
    bits = bf16_matrix(96, 160, seed=11)
    c1, s1 = oracle.per_block_cast(bits, 160, 32, oracle.FMT_E4M3, mode)
    c2, s2 = oracle.per_block_cast(np.ascontiguousarray(bits.T), 96, 32,
                                   oracle.FMT_E4M3, mode)
    assert np.array_equal(c1, c2.T)
    e1 = np.stack([scale_entries(r, 5, mname) for r in s1])
    e2 = np.stack([scale_entries(r, 3, mname) for r in s2])
    assert np.array_equal(e1, e2.T)


@pytest.mark.parametrize("fname,fmt", FMTS)
def test_special_blocks(fname, fmt):
    """All-zero block: the floor scale 1e-4/fmt_max and zero codes; a block
    holding the BF16 maximum: UE8M0 byte 247 (E4M3) / 253 (E2M1); in fp32
    mode every block with amax >= 1e-4 reaches +-fmt_max exactly."""
    bits = bf16_matrix(64, 64, seed=3)
    bits[:32, :32] = 0
    bits[:32, 32:] = 0x7F7F                            # BF16 max
    c, s = oracle.per_block_cast(bits, 64, 32, fmt, oracle.SCALE_FP32)
    assert s[0, 0] == np.float32(np.float32(1e-4) / np.float32(FMT_MAX[fname]))
    assert not unpack(c, fname)[:32, :32].any()
    _, e = oracle.per_block_cast(bits, 64, 32, fmt, oracle.SCALE_UE8M0)
    assert e.view(np.uint8)[0, 1] == (247 if fname == "e4m3" else 253)
    vals = np.abs(decode(unpack(c, fname), fname))
    for rb in range(2):
        for cb in range(2):
            blk = vals[32 * rb:32 * rb + 32, 32 * cb:32 * cb + 32]
            if (rb, cb) != (0, 0):
                assert blk.max() == FMT_MAX[fname]


def test_column_extremes():
    """A zero column takes the floor scale; a column whose amax is exactly
    448 gets s = 1 and codes RNE(x)."""
    bits = bf16_matrix(20, 16, seed=9)
    bits[:, 3] = 0
    col = as_f32(bits[:, 5]).astype(np.float64)
    col = col / np.abs(col).max() * 448.0
    bits[:, 5] = (col.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits[0, 5] = np.float32(448.0).view(np.uint32) >> 16
    x5 = as_f32(bits[:, 5])
    bits[np.abs(x5) > 448, 5] = np.float32(440.0).view(np.uint32) >> 16
    c, s = oracle.per_channel_cast(bits, 16, oracle.FMT_E4M3, oracle.SCALE_FP32)
    assert s[3] == np.float32(np.float32(1e-4) / np.float32(448))
    assert not c[:, 3].any()
    assert s[5] == 1.0
    assert np.array_equal(c[:, 5], nearest_code(as_f32(bits[:, 5]), "e4m3"))


@pytest.mark.parametrize("fname,fmt", FMTS)
def test_pads_and_untouched_memory(fname, fmt):
    """Unused bytes of the last packed word are zero; code-row and scale-row
    stride padding keeps its prior contents."""
    M, K, block = 40, 80, 16                           # 5 block columns
    bits = bf16_matrix(M, K, seed=21)
    rb = K if fname == "e4m3" else K // 2
    codes = np.full((M, rb + 16), 0xA5, np.uint8)
    scales = np.full((3, 4), 0x5A5A5A5A, np.int32)     # 2 words used per row
    oracle.per_block_cast(bits, K, block, fmt, oracle.SCALE_UE8M0,
                          codes=codes[:, :rb], scales=scales[:, :3])
    b = scales.view(np.uint8).reshape(3, 16)
    assert (b[:, 5:8] == 0).all()                      # pad bytes of word 1
    assert (scales[:, 2:] == 0x5A5A5A5A).all()         # beyond the used words
    assert (codes[:, rb:] == 0xA5).all()
    v = np.full(6, 0x5A5A5A5A, np.int32)
    c2 = np.full((M, rb), 0, np.uint8)
    oracle.per_channel_cast(bits, 18, fmt,
                            oracle.SCALE_UE8M0, codes=c2, scales=v[:5])
    vb = v.view(np.uint8)
    assert (vb[18:20] == 0).all() and (v[5] == 0x5A5A5A5A)


def test_thread_split_does_not_change_results():
    bits = bf16_matrix(50, 200, seed=4)
    for fmt in (oracle.FMT_E4M3, oracle.FMT_E2M1):
        a = oracle.per_channel_cast(bits, 200, fmt, oracle.SCALE_UE8M0, threads=1)
        b = oracle.per_channel_cast(bits, 200, fmt, oracle.SCALE_UE8M0, threads=7)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        a = oracle.per_block_cast(bits, 200, 16, fmt, oracle.SCALE_FP32, threads=1)
        b = oracle.per_block_cast(bits, 200, 16, fmt, oracle.SCALE_FP32, threads=3)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_per_channel_without_rows_writes_nothing():
    codes = np.zeros((0, 16), np.uint8)
    s = np.full(16, 7.0, np.float32)
    oracle.per_channel_cast(np.zeros((0, 16), np.uint16), 16, oracle.FMT_E4M3,
                            oracle.SCALE_FP32, codes=codes, scales=s)
    assert (s == 7.0).all()


# ------------------------------------------------------- dequantization

def _codes_without_nan(rng, M, K, fname):
    nb = K if fname == "e4m3" else K // 2
    c = rng.integers(0, 256, size=(M, nb), dtype=np.uint8)
    if fname == "e4m3":
        c[(c & 0x7F) == 0x7F] = 0x35
    return c


def _scale_words(rng, n_rows, n, mname):
    """Random scale rows: positive fp32 values spanning many binades, or
    UE8M0 bytes 1..254 packed four per word (unused bytes zero)."""
    if mname == "ue8m0":
        b = np.zeros((n_rows, -(-n // 4) * 4), np.uint8)
        b[:, :n] = rng.integers(1, 255, size=(n_rows, n), dtype=np.uint8)
        return b.view(np.int32), b[:, :n].astype(np.float64)
    v = np.exp2(rng.uniform(-30, 30, size=(n_rows, n))).astype(np.float32)
    return v, v.astype(np.float64)


def _want(vals, bf16_out):
    y = vals.astype(np.float32)            # the exact product, rounded once
    if bf16_out:
        from precision_quantization_token_gb300.inputs import f32_to_bf16_bits
        return f32_to_bf16_bits(y)
    return y


@pytest.mark.parametrize("fname,fmt", FMTS)
@pytest.mark.parametrize("mname,mode", [("fp32", oracle.SCALE_FP32),
                                        ("ue8m0", oracle.SCALE_UE8M0)])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_block_dequant_is_one_multiply(fname, fmt, mname, mode, bf16_out):
    M, K, block = 70, 96, 32
    rng = np.random.default_rng(31)
    codes = _codes_without_nan(rng, M, K, fname)
    words, sval = _scale_words(rng, -(-M // block), -(-K // block), mname)
    if mname == "ue8m0":
        sval = np.exp2(sval - 127)
    y = oracle.per_block_dequant(codes, words, K, block, fmt, mode,
                                 out_fp32=not bf16_out)
    from bruteforce import decode
    v = decode(unpack(codes, fname), fname)
    s = sval[np.arange(M)[:, None] // block, np.arange(K)[None, :] // block]
    assert np.array_equal(y.view(np.uint16 if bf16_out else np.uint32),
                          _want(v * s, bf16_out).view(np.uint16 if bf16_out else np.uint32))


@pytest.mark.parametrize("fname,fmt", FMTS)
@pytest.mark.parametrize("mname,mode", [("fp32", oracle.SCALE_FP32),
                                        ("ue8m0", oracle.SCALE_UE8M0)])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_channel_dequant_is_one_multiply(fname, fmt, mname, mode, bf16_out):
    M, K = 33, 80
    rng = np.random.default_rng(32)
    codes = _codes_without_nan(rng, M, K, fname)
    words, sval = _scale_words(rng, 1, K, mname)
    if mname == "ue8m0":
        sval = np.exp2(sval - 127)
    y = oracle.per_channel_dequant(codes, words[0], K, fmt, mode,
                                   out_fp32=not bf16_out)
    from bruteforce import decode
    v = decode(unpack(codes, fname), fname)
    assert np.array_equal(y.view(np.uint16 if bf16_out else np.uint32),
                          _want(v * sval[0][None, :], bf16_out).view(
                              np.uint16 if bf16_out else np.uint32))


@pytest.mark.parametrize("fname,fmt", FMTS)
@pytest.mark.parametrize("mname,mode", MODES)
def test_one_row_block_dequant_is_per_token_dequant(fname, fmt, mname, mode):
    K = 5 * 32
    bits = bf16_matrix(1, K, seed=33)
    codes, scales = oracle.per_block_cast(bits, K, 32, fmt, mode)
    a = oracle.per_block_dequant(codes, scales, K, 32, fmt, mode)
    b = oracle.per_token_dequant(codes, scales, K, 32, fmt, mode,
                                 oracle.LAYOUT_ROW_MAJOR)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("fname,fmt", FMTS)
@pytest.mark.parametrize("mname,mode", MODES)
def test_dequant_inverts_the_cast_within_half_a_step(fname, fmt, mname, mode):
    """|x - dequant(cast(x))| <= half the code gap at the decoded value,
    times the scale, plus |x| 2^-23 (the fp32 quotient's rounding)."""
    from bruteforce import decode_table
    M, K = 150, 272
    bits = bf16_matrix(M, K, seed=34)
    x = as_f32(bits).astype(np.float64)
    table = decode_table(fname)
    gaps = np.diff(table)
    for kind in ("block", "channel"):
        if kind == "block":
            codes, scales = oracle.per_block_cast(bits, K, 128, fmt, mode)
            y = oracle.per_block_dequant(codes, scales, K, 128, fmt, mode,
                                         out_fp32=True).astype(np.float64)
        else:
            codes, scales = oracle.per_channel_cast(bits, K, fmt, mode)
            y = oracle.per_channel_dequant(codes, scales, K, fmt, mode,
                                           out_fp32=True).astype(np.float64)
        v = decode(unpack(codes, fname), fname)
        s = np.divide(y, v, out=np.zeros_like(y), where=v != 0)
        # the scale of each element: recover it from a nonzero neighbour's
        # ratio is fragile; bound with the largest gap of the format instead
        # where the code is zero
        idx = np.searchsorted(table, np.abs(v))
        gap = np.where(idx < gaps.size, gaps[np.minimum(idx, gaps.size - 1)],
                       gaps[-1])
        bound = 0.5 * gap * np.abs(s) + np.abs(x) * 2.0 ** -23
        ok = (v == 0) | (np.abs(x - y) <= bound * (1 + 1e-12))
        assert ok.all(), (kind, np.argwhere(~ok)[:3])
