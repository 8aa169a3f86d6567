"""Parity of the per-block and per-channel casts with the oracle (GPU).

The CUDA path is called through the C ABI on guard-banded buffers (a
sentinel row above and below the codes and the scales, sentinel stride
padding, a poisoned input stride pad); the oracle runs on the same host
bytes; codes, scales and every sentinel must agree bit for bit.
"""
import numpy as np
import pytest

import oracle
import precision_quantization_token_gb300 as tk
from gpu_util import FMT_ID, MODE_ID, THREADS, torch_mod
from precision_quantization_token_gb300.inputs import (WORKLOADS, make_input,
                                                       random_bf16)

pytestmark = pytest.mark.gpu

SENT_CODE = 0xA5
SENT_WORD = 0x5A5A5A5A
POISON_BF16 = 0x7F00
FMTS = ["e4m3", "e2m1"]
MODES = ["fp32", "pow2", "ue8m0"]


def _host_x(bits, ld_x):
    M, K = bits.shape
    x = np.full((M, ld_x), POISON_BF16, np.uint16)
    x[:, :K] = bits
    return x


def _stream():
    return torch_mod().cuda.current_stream().cuda_stream


def _dev(a, dtype_view=None):
    torch = torch_mod()
    return torch.from_numpy(a.view(dtype_view) if dtype_view else a).cuda()


def _row_bytes(K, fmt):
    return K if fmt == "e4m3" else K // 2


def run_block(bits, fmt, mode, ld_x=None, code_pad=0, scale_pad=0):
    """(gpu codes, gpu scales, oracle codes, oracle scales), guards included."""
    torch = torch_mod()
    M, K = bits.shape
    ld_x = ld_x or K
    x = _host_x(bits, ld_x)
    rb = _row_bytes(K, fmt)
    ld_codes = (rb + code_pad + 15) // 16 * 16
    nr, nw, _ = oracle.block_scale_shape(M, K, 128, MODE_ID[mode])
    ld_s = nw + scale_pad
    codes = np.full((M + 2, ld_codes), SENT_CODE, np.uint8)
    scales = np.full((nr + 2, ld_s), SENT_WORD, np.uint32)

    xd, cd, sd = _dev(x, np.int16), _dev(codes), _dev(scales, np.int32)
    tk.tk_per_block_cast(xd.data_ptr(), M, K, ld_x, tk.FMT[fmt],
                         tk.SCALE[mode], cd.data_ptr() + ld_codes, ld_codes,
                         sd.data_ptr() + 4 * ld_s, ld_s, _stream())
    torch.cuda.synchronize()
    gc, gs = cd.cpu().numpy(), sd.cpu().numpy().view(np.uint32)

    rc, rs = codes.copy(), scales.copy()
    s_view = rs[1:nr + 1].view(np.int32 if mode == "ue8m0" else np.float32)
    if M:
        oracle.per_block_cast(x, K, 128, FMT_ID[fmt], MODE_ID[mode],
                              codes=rc[1:M + 1], scales=s_view,
                              threads=THREADS)
    return gc, gs, rc, rs


def run_channel(bits, fmt, mode, ld_x=None, code_pad=0, workspace=None):
    torch = torch_mod()
    M, K = bits.shape
    ld_x = ld_x or K
    x = _host_x(bits, ld_x)
    rb = _row_bytes(K, fmt)
    ld_codes = (rb + code_pad + 15) // 16 * 16
    nw, _ = oracle.channel_scale_shape(K, MODE_ID[mode])
    codes = np.full((M + 2, ld_codes), SENT_CODE, np.uint8)
    scales = np.full(nw + 8, SENT_WORD, np.uint32)      # 4 guard words each side

    xd, cd, sd = _dev(x, np.int16), _dev(codes), _dev(scales, np.int32)
    need = tk.tk_per_channel_workspace_bytes(K)
    if workspace is None:     # zero-filled before first use
        workspace = torch.zeros(need + 64, dtype=torch.uint8, device="cuda")[:need]
    tk.tk_per_channel_cast(xd.data_ptr(), M, K, ld_x, tk.FMT[fmt],
                           tk.SCALE[mode], cd.data_ptr() + ld_codes, ld_codes,
                           sd.data_ptr() + 16, workspace.data_ptr(),
                           workspace.numel(), _stream())
    torch.cuda.synchronize()
    gc, gs = cd.cpu().numpy(), sd.cpu().numpy().view(np.uint32)
    # every completed call leaves the workspace zero-filled
    assert not workspace.cpu().numpy().any(), "workspace not left zero-filled"

    rc, rs = codes.copy(), scales.copy()
    s_view = rs[4:4 + nw].view(np.int32 if mode == "ue8m0" else np.float32)
    if M:
        oracle.per_channel_cast(x, K, FMT_ID[fmt], MODE_ID[mode],
                                codes=rc[1:M + 1], scales=s_view,
                                threads=THREADS)
    return gc, gs, rc, rs


def assert_same(gc, gs, rc, rs):
    if not np.array_equal(gc, rc):
        bad = np.argwhere(gc != rc)
        r, c = bad[0]
        raise AssertionError(f"codes differ at {bad.shape[0]} bytes; first "
                             f"(row {r - 1}, byte {c}): gpu {gc[r, c]:#04x} "
                             f"oracle {rc[r, c]:#04x}")
    if not np.array_equal(gs, rs):
        bad = np.argwhere(gs != rs)
        raise AssertionError(f"scales differ at {bad.shape[0]} words; first "
                             f"{bad[0]}: gpu {gs[tuple(bad[0])]:#010x} oracle "
                             f"{rs[tuple(bad[0])]:#010x}")


def bits_with_specials(M, K, seed):
    """Normal values spread over rows and columns, plus exact zero blocks /
    columns, -0, BF16 denormals and the BF16 maximum."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((M, K)).astype(np.float32)
    v *= np.exp2(rng.integers(-8, 9, (M, 1))).astype(np.float32)
    v *= np.exp2(rng.integers(-6, 7, (1, K))).astype(np.float32)
    bits = (v.view(np.uint32) >> 16).astype(np.uint16)
    bits[rng.random((M, K)) < 0.02] = 0x8000                   # -0
    den = rng.random((M, K)) < 0.01
    bits[den] = (rng.integers(1, 128, den.sum()) |
                 (rng.integers(0, 2, den.sum()) << 15)).astype(np.uint16)
    if M > 130 and K > 140:
        bits[:128, :128] = 0                                   # a zero block
        bits[128:, 3] = 0                                      # zero column tail
        bits[129, 137] = 0x7F7F                                # BF16 max
        bits[130, 138] = 0xFF7F                                # -BF16 max
    return bits


# ---------------------------------------------------------------- full size

@pytest.mark.parametrize("name", ["pb2", "pc2"])
def test_full_workload(name):
    w = WORKLOADS[name]
    bits = make_input(w)
    run = run_block if w.op == "block" else run_channel
    assert_same(*run(bits, w.fmt, w.scale))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", MODES)
def test_full_shape_every_option(fmt, mode):
    bits = make_input(WORKLOADS["c2"], M=1024)
    assert_same(*run_block(bits, fmt, mode))
    assert_same(*run_channel(bits, fmt, mode))


# ------------------------------------------------------------------ shapes

SHAPES = [(1, 16), (1, 128), (127, 128), (128, 256), (129, 272), (300, 400),
          (255, 2064), (640, 7184), (2, 4096)]


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", MODES)
def test_block_shapes(M, K, fmt, mode):
    assert_same(*run_block(bits_with_specials(M, K, seed=M * 7 + K), fmt, mode))


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", MODES)
def test_channel_shapes(M, K, fmt, mode):
    assert_same(*run_channel(bits_with_specials(M, K, seed=M * 5 + K), fmt,
                             mode))


@pytest.mark.parametrize("fmt", FMTS)
def test_strides_and_pads(fmt):
    bits = bits_with_specials(300, 400, seed=3)
    assert_same(*run_block(bits, fmt, "ue8m0", ld_x=424, code_pad=32,
                           scale_pad=3))
    assert_same(*run_block(bits, fmt, "fp32", ld_x=408, code_pad=16,
                           scale_pad=1))
    assert_same(*run_channel(bits, fmt, "fp32", ld_x=416, code_pad=48))


def test_tall_columns():
    """Many row tiles fold into each column amax (atomics across CTAs)."""
    bits = random_bf16(8, 70000, 48)
    bits[69999, 5] = 0x4600                                    # lone max, last row
    bits[0, 6] = 0xC600                                        # lone -max, first row
    for mode in MODES:
        assert_same(*run_channel(bits, "e4m3", mode))


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bf16_value(fmt):
    """All 65,280 finite BF16 patterns (a 256 x 256 matrix with the NaN/Inf
    patterns replaced by zero): every value passes through both casts."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    bits[exp == 0xFF] = 0
    bits = bits.reshape(256, 256)
    for mode in MODES:
        assert_same(*run_block(bits, fmt, mode))
        assert_same(*run_channel(bits, fmt, mode))
        assert_same(*run_channel(np.ascontiguousarray(bits.T), fmt, mode))


def test_workspace_reused_across_calls():
    """Calls in a row on one workspace, with different shapes: none sees an
    earlier call's column maxima, and each leaves the workspace zero."""
    torch = torch_mod()
    ws = torch.zeros(tk.tk_per_channel_workspace_bytes(4096), dtype=torch.uint8,
                     device="cuda")
    big = random_bf16(1, 200, 512, scale=100.0)
    small = random_bf16(2, 200, 512, scale=0.01)
    assert_same(*run_channel(big, "e4m3", "fp32", workspace=ws))
    assert_same(*run_channel(small, "e4m3", "fp32", workspace=ws))
    assert_same(*run_channel(random_bf16(3, 1000, 4096), "e2m1", "ue8m0",
                             workspace=ws))
    assert_same(*run_channel(random_bf16(4, 7, 160, scale=1e-3), "e4m3",
                             "pow2", workspace=ws))
    assert_same(*run_channel(big, "e4m3", "fp32", workspace=ws))


def test_empty_batch_is_a_noop():
    torch = torch_mod()
    s = _stream()
    tk.tk_per_block_cast(0, 0, 256, 256, 0, 0, 0, 256, 0, 2, s)
    tk.tk_per_channel_cast(0, 0, 256, 256, 0, 0, 0, 256, 0, 0,
                           tk.tk_per_channel_workspace_bytes(256), s)
    torch.cuda.synchronize()


def test_tensor_api():
    torch = torch_mod()
    bits = make_input(WORKLOADS["c2"], M=512)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    for fmt in FMTS:
        for mode in MODES:
            c, s = tk.per_block_cast(x, fmt, mode)
            rc, rs = oracle.per_block_cast(bits, 7168, 128, FMT_ID[fmt],
                                           MODE_ID[mode], threads=THREADS)
            assert np.array_equal(c.cpu().numpy(), rc)
            assert np.array_equal(s.cpu().numpy().view(np.uint32),
                                  rs.view(np.uint32))
            c, s = tk.per_channel_cast(x, fmt, mode)
            rc, rs = oracle.per_channel_cast(bits, 7168, FMT_ID[fmt],
                                             MODE_ID[mode], threads=THREADS)
            assert np.array_equal(c.cpu().numpy(), rc)
            assert np.array_equal(s.cpu().numpy().view(np.uint32),
                                  rs.view(np.uint32))


def test_zz_no_tile_kernel_gave_up_on_a_wait():
    assert tk.tk_get_device_fault(clear=False) == 0


# ------------------------------------------------- per-block / per-channel
# dequantization: bit-exact against the oracle on the same host codes and
# scales (from the oracle's casts, and random codes with every scale byte)

def _run_dequant(kind, codes, scales, M, K, fmt, mode, out, ld_y=None):
    torch = torch_mod()
    rb = _row_bytes(K, fmt)
    ld_codes = codes.shape[1]
    assert ld_codes % 16 == 0 and ld_codes >= rb
    ld_y = ld_y or K
    esz = 4 if out == "fp32" else 2
    y = np.full((M + 2, ld_y * esz), 0xA5, np.uint8)
    cd = _dev(np.ascontiguousarray(codes))
    sd = _dev(np.ascontiguousarray(scales).view(np.uint8))
    yd = _dev(y)
    if kind == "block":
        tk.tk_per_block_dequant(cd.data_ptr(), ld_codes, sd.data_ptr(),
                                scales.shape[1], M, K, tk.FMT[fmt],
                                tk.SCALE[mode], yd.data_ptr() + ld_y * esz,
                                ld_y, tk.OUT_DTYPE[out], _stream())
    else:
        tk.tk_per_channel_dequant(cd.data_ptr(), ld_codes, sd.data_ptr(), M,
                                  K, tk.FMT[fmt], tk.SCALE[mode],
                                  yd.data_ptr() + ld_y * esz, ld_y,
                                  tk.OUT_DTYPE[out], _stream())
    torch.cuda.synchronize()
    g = yd.cpu().numpy()
    ref = y.copy()
    if kind == "block":
        yo = oracle.per_block_dequant(codes, scales, K, 128, FMT_ID[fmt],
                                      MODE_ID[mode], out_fp32=out == "fp32",
                                      threads=THREADS)
    else:
        yo = oracle.per_channel_dequant(codes, scales.reshape(-1), K,
                                        FMT_ID[fmt], MODE_ID[mode],
                                        out_fp32=out == "fp32", threads=THREADS)
    ref[1:M + 1, :K * esz] = yo.view(np.uint8).reshape(M, K * esz)
    return g, ref


def _padded_codes(codes, K, fmt):
    rb = _row_bytes(K, fmt)
    ld = (rb + 15) // 16 * 16
    out = np.zeros((codes.shape[0], ld), np.uint8)
    out[:, :rb] = codes[:, :rb]
    return out


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_dequant_of_the_casts(fmt, mode, out):
    M, K = 1000, 7184
    bits = bits_with_specials(M, K, seed=41)
    fid, mid = FMT_ID[fmt], MODE_ID[mode]
    codes, scales = oracle.per_block_cast(bits, K, 128, fid, mid, threads=THREADS)
    g, r = _run_dequant("block", _padded_codes(codes, K, fmt), scales, M, K,
                        fmt, mode, out)
    assert np.array_equal(g, r)
    codes, scales = oracle.per_channel_cast(bits, K, fid, mid, threads=THREADS)
    sv = np.zeros(-(-scales.size // 4) * 4, scales.dtype)  # 16-byte multiple
    sv[:scales.size] = scales
    g, r = _run_dequant("channel", _padded_codes(codes, K, fmt), sv, M, K,
                        fmt, mode, out)
    assert np.array_equal(g, r)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", ["fp32", "ue8m0"])
def test_dequant_every_code_and_scale(fmt, mode):
    """Random code bytes (no NaN codes) under every UE8M0 byte 0..254 (0 is
    the denormal 2^-127; 255, +inf, makes 0 * inf NaNs whose bit patterns
    are not defined), or fp32 scales over a wide range."""
    rng = np.random.default_rng(42)
    M, K = 256, 1024
    codes = rng.integers(0, 256, size=(M, _row_bytes(K, fmt)), dtype=np.uint8)
    if fmt == "e4m3":
        codes[(codes & 0x7F) == 0x7F] = 0x11
    codes = _padded_codes(codes, K, fmt)
    if mode == "ue8m0":
        blk = rng.integers(0, 255, size=(2, 8), dtype=np.uint8)
        blk.reshape(-1)[:2] = (0, 254)
        bs = blk.view(np.int32)
        ch = (np.arange(K, dtype=np.uint32) % 255).astype(np.uint8)  # 0..254
        cs = ch.view(np.int32)
    else:
        bs = np.exp2(rng.uniform(-40, 40, size=(2, 8))).astype(np.float32)
        cs = np.exp2(rng.uniform(-40, 40, size=K)).astype(np.float32)
    for out in ("bf16", "fp32"):
        g, r = _run_dequant("block", codes, bs, M, K, fmt, mode, out)
        assert np.array_equal(g, r)
        g, r = _run_dequant("channel", codes, cs, M, K, fmt, mode, out)
        assert np.array_equal(g, r)


def test_dequant_strided_output_and_tensor_api():
    torch = torch_mod()
    M, K = 300, 400
    bits = bits_with_specials(M, K, seed=43)
    codes, scales = oracle.per_block_cast(bits, K, 128, oracle.FMT_E4M3,
                                          oracle.SCALE_FP32)
    g, r = _run_dequant("block", _padded_codes(codes, K, "e4m3"), scales, M, K,
                        "e4m3", "fp32", "bf16", ld_y=424)
    assert np.array_equal(g, r)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    for fmt in FMTS:
        c, s = tk.per_channel_cast(x, fmt, "ue8m0")
        y = tk.per_channel_dequant(c, s, K, fmt, "ue8m0", out_dtype="fp32")
        rc, rs = oracle.per_channel_cast(bits, K, FMT_ID[fmt], oracle.SCALE_UE8M0)
        yo = oracle.per_channel_dequant(rc, rs, K, FMT_ID[fmt],
                                        oracle.SCALE_UE8M0, out_fp32=True)
        assert np.array_equal(y.cpu().numpy().view(np.uint32), yo.view(np.uint32))
        c, s = tk.per_block_cast(x, fmt, "pow2")
        y = tk.per_block_dequant(c, s, K, fmt, "pow2")
        rc, rs = oracle.per_block_cast(bits, K, 128, FMT_ID[fmt],
                                       oracle.SCALE_FP32_POW2)
        yo = oracle.per_block_dequant(rc, rs, K, 128, FMT_ID[fmt],
                                      oracle.SCALE_FP32_POW2)
        assert np.array_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), yo)


def test_zz_dequant_fault_word_clear():
    assert tk.tk_get_device_fault(clear=False) == 0


# ------------------------------------------------------------ large index

def _tiled_device_matrix(torch, block, M):
    """A device [M, K] int16 matrix repeating the host block's rows."""
    K = block.shape[1]
    dev_block = torch.from_numpy(block.view(np.int16)).cuda()
    x = torch.empty((M, K), dtype=torch.int16, device="cuda")
    for r0 in range(0, M, block.shape[0]):
        n = min(block.shape[0], M - r0)
        x[r0:r0 + n] = dev_block[:n]
    return x


def test_per_block_beyond_2_31_elements():
    """More than 2^31 elements (64-bit addressing): the input repeats a
    1,152-row host block (9 block rows), so block row i equals host block
    row i mod 9; sampled block rows on both sides of 2^31 elements are
    checked against the oracle's cast of the host block."""
    torch = torch_mod()
    K, hb = 16384, 1152
    M = -(-((1 << 31) // K + 1000) // 128) * 128
    block = random_bf16(124, hb, K, scale=3.0)
    x = _tiled_device_matrix(torch, block, M)
    n_cb = K // 128
    codes = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    scales = torch.empty((M // 128, n_cb), dtype=torch.float32, device="cuda")
    tk.tk_per_block_cast(x.data_ptr(), M, K, K, 0, 0, codes.data_ptr(), K,
                         scales.data_ptr(), n_cb, _stream())
    torch.cuda.synchronize()
    rc, rs = oracle.per_block_cast(block, K, 128, oracle.FMT_E4M3,
                                   oracle.SCALE_FP32, threads=THREADS)
    edge = (1 << 31) // K // 128                       # block row at 2^31
    for bi in sorted({0, 1, edge - 1, edge, edge + 1, M // 128 - 1}):
        lo = (bi % (hb // 128)) * 128
        got = codes[bi * 128:(bi + 1) * 128].cpu().numpy()
        assert np.array_equal(got, rc[lo:lo + 128]), bi
        assert np.array_equal(scales[bi].cpu().numpy().view(np.uint32),
                              rs[bi % (hb // 128)].view(np.uint32)), bi
    del x, codes, scales
    torch.cuda.empty_cache()


def test_per_channel_beyond_2_31_elements():
    """More than 2^31 elements: the input repeats a 999-row host block, and
    the last row (past 2^31 elements) holds outliers in some columns, so
    every column maximum and hence every scale depends on rows the 32-bit
    offsets could not reach."""
    torch = torch_mod()
    K, hb = 16384, 999
    M = (1 << 31) // K + 1000
    block = random_bf16(125, hb, K)
    x = _tiled_device_matrix(torch, block, M)
    last = np.zeros((1, K), np.uint16)
    last[0, ::7] = 0x4480                                  # 1024, a new column max
    x[M - 1] = torch.from_numpy(last.view(np.int16)).cuda()[0]
    codes = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    scales = torch.empty(K, dtype=torch.float32, device="cuda")
    ws = torch.zeros(tk.tk_per_channel_workspace_bytes(K), dtype=torch.uint8,
                     device="cuda")
    tk.tk_per_channel_cast(x.data_ptr(), M, K, K, 0, 0, codes.data_ptr(), K,
                           scales.data_ptr(), ws.data_ptr(), ws.numel(),
                           _stream())
    torch.cuda.synchronize()
    host = np.vstack([block, last])
    rc, rs = oracle.per_channel_cast(host, K, oracle.FMT_E4M3,
                                     oracle.SCALE_FP32, threads=THREADS)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32),
                          rs.view(np.uint32))
    edge = (1 << 31) // K
    sample = sorted({0, 1, M // 2, edge - 1, edge, edge + 1, M - 2})
    idx = torch.tensor(sample, device="cuda")
    got = codes.index_select(0, idx).cpu().numpy()
    for i, m in enumerate(sample):
        assert np.array_equal(got[i], rc[m % hb]), m
    assert np.array_equal(codes[M - 1].cpu().numpy(), rc[hb])
    assert not ws.cpu().numpy().any()
    del x, codes, scales
    torch.cuda.empty_cache()


def test_zz_large_index_fault_word_clear():
    assert tk.tk_get_device_fault(clear=False) == 0
