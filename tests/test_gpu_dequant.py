"""GPU parity of per-token dequantization and cast-and-cast-back, through
the C ABI, against the oracle (bit-exact, BF16 and fp32 outputs).  Codes and
scales fed to the dequantization are written by the oracle's cast."""
import zlib

import numpy as np
import pytest

import oracle
import precision_quantization_token_gb300 as tk
from gpu_util import THREADS
from precision_quantization_token_gb300.inputs import (WORKLOADS, make_input,
                                                       random_bf16)

pytestmark = pytest.mark.gpu

FMT = {"e4m3": oracle.FMT_E4M3, "e2m1": oracle.FMT_E2M1}
MODE = {"fp32": oracle.SCALE_FP32, "pow2": oracle.SCALE_FP32_POW2,
        "ue8m0": oracle.SCALE_UE8M0}
LAYOUT = {"row": oracle.LAYOUT_ROW_MAJOR, "transposed": oracle.LAYOUT_TRANSPOSED}
GUARD = 0x5A5A


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    import torch
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    tk.build()
    tk.load()
    yield


def gpu_dequant(codes, scales, K, group, fmt, mode, layout, out="bf16",
                ld_y=None):
    """Run the CUDA dequantization on host arrays (guard rows around y)."""
    import torch
    M = codes.shape[0]
    ld_y = ld_y or K
    esize = 2 if out == "bf16" else 4
    y = torch.full(((M + 2) * ld_y * esize // 2,), GUARD, dtype=torch.int16,
                   device="cuda")
    cd = torch.from_numpy(np.ascontiguousarray(codes)).cuda()
    sd = torch.from_numpy(np.ascontiguousarray(scales).view(np.int32)).cuda()
    tk.tk_per_token_dequant(cd.data_ptr(), cd.stride(0), sd.data_ptr(),
                            sd.stride(0), M, K, group, tk.FMT[fmt],
                            tk.SCALE[mode], tk.LAYOUT[layout],
                            y.data_ptr() + ld_y * esize, ld_y,
                            tk.OUT_DTYPE[out],
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    raw = y.cpu().numpy().view(np.uint16 if out == "bf16" else np.uint32)
    raw = raw.reshape(M + 2, ld_y)
    assert np.all(raw[0].view(np.uint16) == GUARD)
    assert np.all(raw[-1].view(np.uint16) == GUARD)
    if ld_y > K:
        assert np.all(raw[1:-1, K:].view(np.uint16) == GUARD)
    return raw[1:-1, :K]


def oracle_dequant(codes, scales, K, group, fmt, mode, layout, out="bf16"):
    y = oracle.per_token_dequant(codes, scales, K, group, FMT[fmt], MODE[mode],
                                 LAYOUT[layout], out_fp32=(out == "fp32"),
                                 threads=THREADS)
    return y if out == "bf16" else y.view(np.uint32)


def oracle_codes(bits, K, group, fmt, mode, layout):
    """Codes and scales written by the oracle's cast, code rows padded to a
    16-byte stride (the alignment the library requires)."""
    row_bytes = K if fmt == "e4m3" else K // 2
    codes = np.zeros((bits.shape[0], -(-row_bytes // 16) * 16), np.uint8)
    return oracle.per_token_cast(bits, K, group, FMT[fmt], MODE[mode],
                                 LAYOUT[layout], codes=codes, threads=THREADS)


@pytest.mark.parametrize("name", ["c2", "c3a", "c5"])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_dequant_full_workload(name, out):
    w = WORKLOADS[name]
    bits = make_input(w)
    codes, scales = oracle_codes(bits, w.K, w.group, w.fmt, w.scale, w.layout)
    got = gpu_dequant(codes, scales, w.K, w.group, w.fmt, w.scale, w.layout,
                      out)
    want = oracle_dequant(codes, scales, w.K, w.group, w.fmt, w.scale,
                          w.layout, out)
    assert np.array_equal(got, want)


def _shape_cases():
    out = []
    for fmt in ("e4m3", "e2m1"):
        for mode in ("fp32", "ue8m0"):
            for layout in ("row", "transposed"):
                for M, K, group in [(1, 16, 16), (3, 48, 16), (254, 272, 16),
                                    (5, 1040, 16), (33, 7168, 128),
                                    (7, 16512, 128), (130, 4096, 32)]:
                    out.append((fmt, mode, layout, M, K, group))
    return out


@pytest.mark.parametrize("fmt,mode,layout,M,K,group", _shape_cases())
def test_dequant_shapes(fmt, mode, layout, M, K, group):
    seed = zlib.crc32(repr((fmt, mode, layout, M, K)).encode()) & 0xFFFF
    bits = random_bf16(seed, M, K, scale=3.0)
    codes, scales = oracle_codes(bits, K, group, fmt, mode, layout)
    for out in ("bf16", "fp32"):
        got = gpu_dequant(codes, scales, K, group, fmt, mode, layout, out,
                          ld_y=K + 8 if out == "bf16" else K + 4)
        want = oracle_dequant(codes, scales, K, group, fmt, mode, layout, out)
        assert np.array_equal(got, want), (out,)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "ue8m0"])
def test_dequant_every_code_and_scale(fmt, mode):
    """Every code value against a spread of scales: fp32 scales across the
    exponent range, or every UE8M0 byte 1..254 plus 0 (2^-127, denormal)."""
    rng = np.random.default_rng(17)
    M, group = 256, 16
    K = 16 * 16
    if fmt == "e4m3":
        c = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
        codes = rng.choice(c, size=(M, K)).astype(np.uint8)
    else:
        nib = rng.integers(0, 16, size=(M, K), dtype=np.uint8)
        codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    G = K // group
    if mode == "ue8m0":
        e = rng.integers(0, 255, size=(M, G), dtype=np.uint8)
        e[0, :] = 0
        scales = np.ascontiguousarray(e).view(np.int32)
    else:
        scales = (rng.uniform(1, 2, size=(M, G)) *
                  np.exp2(rng.integers(-140, 120, size=(M, G)))).astype(np.float32)
    for out in ("bf16", "fp32"):
        got = gpu_dequant(codes, scales, K, group, fmt, mode, "row", out)
        want = oracle_dequant(codes, scales, K, group, fmt, mode, "row", out)
        assert np.array_equal(got, want), out


def test_dequant_nan_code_gives_nan():
    codes = np.full((1, 16), 0x7F, np.uint8)
    codes[0, 1] = 0xFF
    scales = np.ones((1, 1), np.float32)
    got = gpu_dequant(codes, scales, 16, 16, "e4m3", "fp32", "row", "fp32")
    assert np.all(np.isnan(got.view(np.float32)))


# --------------------------------------------------------- cast-and-cast-back

def gpu_cast_back(bits, K, group, fmt, mode, ld_x=None, ld_y=None):
    import torch
    M = bits.shape[0]
    ld_x = ld_x or K
    ld_y = ld_y or K
    xh = np.full((M, ld_x), 0x7F00, np.uint16)
    xh[:, :K] = bits
    xd = torch.from_numpy(xh.view(np.int16)).cuda()
    y = torch.full(((M + 2) * ld_y,), GUARD, dtype=torch.int16, device="cuda")
    tk.tk_per_token_cast_back(xd.data_ptr(), M, K, ld_x, group, tk.FMT[fmt],
                              tk.SCALE[mode], y.data_ptr() + ld_y * 2, ld_y,
                              torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    raw = y.cpu().numpy().view(np.uint16).reshape(M + 2, ld_y)
    assert np.all(raw[0] == GUARD) and np.all(raw[-1] == GUARD)
    if ld_y > K:
        assert np.all(raw[1:-1, K:] == GUARD)
    return raw[1:-1, :K]


@pytest.mark.parametrize("name", ["c2", "c3a", "c5"])
def test_cast_back_full_workload(name):
    w = WORKLOADS[name]
    bits = make_input(w)
    got = gpu_cast_back(bits, w.K, w.group, w.fmt, w.scale)
    want = oracle.per_token_cast_back(bits, w.K, w.group, FMT[w.fmt],
                                      MODE[w.scale], threads=THREADS)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "pow2", "ue8m0"])
def test_cast_back_shapes_and_edges(fmt, mode):
    for (M, K, group) in [(1, 16, 16), (3, 48, 16), (254, 1088, 64),
                          (7, 16512, 128), (65, 4096, 32)]:
        bits = random_bf16(M + K, M, K, scale=2.0)
        bits[0, :group] = 0x8000                              # -0 group
        if M > 2:
            bits[1] = 0x7F7F                                  # BF16 max
            bits[2, ::3] = 0x0001                             # denormals
        got = gpu_cast_back(bits, K, group, fmt, mode, ld_x=K + 8,
                            ld_y=K + 16)
        want = oracle.per_token_cast_back(bits, K, group, FMT[fmt], MODE[mode],
                                          threads=THREADS)
        assert np.array_equal(got, want), (M, K, group)


def test_tensor_api_round_trip():
    import torch
    bits = random_bf16(5, 300, 2048)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    codes, scales = tk.per_token_cast(x, group=128, fmt="e4m3", scale="ue8m0",
                                      layout="transposed")
    y = tk.per_token_dequant(codes, scales, 2048, group=128, fmt="e4m3",
                             scale="ue8m0", layout="transposed")
    back = tk.per_token_cast_back(x, group=128, fmt="e4m3", scale="ue8m0")
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), back.view(torch.int16))
