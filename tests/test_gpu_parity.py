"""GPU parity: the CUDA path, called through the C ABI, against the oracle.

Plain cast: bit-exact codes and scales, with guard rows, stride padding and
scale padding checked untouched.  Fused SwiGLU: the tolerance of
gpu_util.check_swiglu.  Run on a GB300 with ``pytest -m gpu``.
"""
import zlib

import numpy as np
import pytest

import oracle
import precision_quantization_token_gb300 as tk
from gpu_util import THREADS, Case, assert_bit_exact, check_swiglu
from precision_quantization_token_gb300.inputs import (WORKLOADS,
                                                       bf16_bits_to_f32,
                                                       f32_to_bf16_bits,
                                                       make_input,
                                                       random_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    import torch
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    tk.build()
    tk.load()
    yield


# ------------------------------------------------------------ full sizes

@pytest.mark.parametrize("name", ["c1", "c2", "c3a", "c3b", "c4", "c5"])
def test_full_workload(name):
    """Every workload at its full size, in the launch configuration the
    benchmark times (the library picks the grid the same way)."""
    w = WORKLOADS[name]
    bits = make_input(w)
    case = Case(bits, w.K, w.group, w.fmt, w.scale, w.layout, swiglu=w.swiglu)
    if w.swiglu:
        stats = check_swiglu(case)
        print(name, stats)
    else:
        assert_bit_exact(case)


# --------------------------------------------------- small, ragged shapes

SHAPES = {16: [16, 48, 272, 1040], 32: [32, 96, 4128], 64: [64, 192, 1088],
          128: [128, 384, 7168]}
ROWS = [1, 3, 5, 254, 1031]


def _small_cases():
    out = []
    for fmt in ("e4m3", "e2m1"):
        for mode in ("fp32", "pow2", "ue8m0"):
            for layout in ("row", "transposed"):
                for group, Ks in SHAPES.items():
                    for i, K in enumerate(Ks):
                        M = ROWS[(i + group // 16 + len(mode)) % len(ROWS)]
                        out.append((fmt, mode, layout, group, K, M))
    return out


@pytest.mark.parametrize("fmt,mode,layout,group,K,M", _small_cases())
def test_small_shapes(fmt, mode, layout, group, K, M):
    seed = zlib.crc32(repr((fmt, mode, layout, group, K, M)).encode()) & 0xFFFF
    bits = random_bf16(seed, M, K, scale=2.0)
    case = Case(bits, K, group, fmt, mode, layout)
    assert_bit_exact(case)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("layout", ["row", "transposed"])
def test_strides_and_padding(fmt, layout):
    """ld_x > K (poisoned pad), code rows and scale rows with spare space."""
    M, K, group = 77, 640, 64
    bits = random_bf16(11, M, K)
    for mode in ("fp32", "ue8m0"):
        case = Case(bits, K, group, fmt, mode, layout, ld_x=K + 24,
                    code_pad=32, scale_pad=3)
        assert_bit_exact(case)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "pow2"])
@pytest.mark.parametrize("group,K", [(16, 256), (16, 512), (32, 512), (32, 1024),
                                     (16, 2048), (32, 4096)])
def test_interleaved_rows_transposed(fmt, mode, group, K):
    """Transposed fp32 / pow2 scales of groups of 16 or 32 with a power of
    two of whole rows per 16 KiB tile (2 to 32): the kernel interleaves a
    full tile's rows over lanes.  Batches of full tiles, with a ragged last
    tile (which takes the plain mapping), and smaller than one tile."""
    rows = 16384 // (2 * K)
    for M in (3 * rows + 1, 2 * rows, max(rows - 1, 1)):
        seed = zlib.crc32(repr((fmt, mode, group, K, M)).encode()) & 0xFFFF
        bits = random_bf16(seed, M, K, scale=2.0)
        assert_bit_exact(Case(bits, K, group, fmt, mode, "transposed"))


@pytest.mark.parametrize("mode", ["fp32", "pow2"])
@pytest.mark.parametrize("group,N", [(32, 256), (16, 512), (32, 1024), (32, 2048)])
def test_interleaved_rows_transposed_swiglu(mode, group, N):
    """The fused SwiGLU cast on row-interleaved tiles (gate and up halves
    share a 16 KiB tile: 2 to 16 rows)."""
    rows = 16384 // (4 * N)
    for M in (3 * rows + 1, 2 * rows):
        bits = random_bf16(N + M + group, M, 2 * N, scale=2.0)
        case = Case(bits, N, group, "e4m3", mode, "transposed", swiglu=True)
        check_swiglu(case, max_code_frac=2e-3 if M * N < 5000 else 1e-4)


def test_empty_batch():
    case = Case(np.zeros((0, 128), np.uint16), 128, 128, "e4m3", "fp32",
                "row")
    assert_bit_exact(case)


# ---------------------------------------------------------- value edges

@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "pow2", "ue8m0"])
def test_exhaustive_unit_scale(fmt, mode):
    """Every BF16 value with |x| <= fmt_max, in groups led by +-fmt_max (scale
    exactly 1), so each code is the hardware rounding of x itself."""
    fmt_max = 448.0 if fmt == "e4m3" else 6.0
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= fmt_max)
    xs = (bits[keep]).astype(np.uint16)
    group = 128
    per = group - 1
    n_groups = -(-xs.size // per)
    pad = np.zeros(n_groups * per, np.uint16)
    pad[:xs.size] = xs
    body = pad.reshape(n_groups, per)
    lead = f32_to_bf16_bits(np.where(np.arange(n_groups) % 2, -fmt_max,
                                     fmt_max).astype(np.float32))
    rows = np.concatenate([lead[:, None], body], axis=1)     # [n_groups, 128]
    K = group * 8
    n_rows = -(-n_groups // 8)
    full = np.zeros((n_rows * 8, group), np.uint16)
    full[:n_groups] = rows
    full[n_groups:, 0] = f32_to_bf16_bits(np.float32(fmt_max))
    bits2d = full.reshape(n_rows, K)
    assert_bit_exact(Case(bits2d, K, group, fmt, mode, "row"))


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "ue8m0"])
def test_special_rows(fmt, mode):
    """Zero rows, -0 rows, denormal rows, BF16 extremes, huge dynamic range
    inside a row, lone outliers."""
    M, K, group = 64, 512, 16 if fmt == "e2m1" else 128
    rng = np.random.default_rng(5)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= (10.0 ** rng.uniform(-30, 30, size=(M, 1))).astype(np.float32)
    bits = f32_to_bf16_bits(x)
    bits[0] = 0
    bits[1] = 0x8000
    bits[2] = rng.integers(1, 128, size=K).astype(np.uint16) | \
        (rng.integers(0, 2, size=K).astype(np.uint16) << 15)
    bits[3] = 0x7F7F                                   # largest BF16
    bits[4] = 0xFF7F                                   # most negative BF16
    bits[5, ::3] = 0x0001                              # smallest denormal
    bits[6] = f32_to_bf16_bits(np.float32(1e-4))
    bits[7, 7] = 0x7F7F                                # one huge outlier
    bits[8] = f32_to_bf16_bits(
        np.float32(1.0) * np.where(np.arange(K) % 2, 1, -1).astype(np.float32))
    bits[9, :] = 0x0080                                # smallest normal
    assert_bit_exact(Case(bits, K, group, fmt, mode, "row"))
    assert_bit_exact(Case(bits, K, group, fmt, mode, "transposed"))


def test_fp32_scale_quotients_across_range():
    """fp32 scales over the whole BF16 exponent range: the quotient from the
    reciprocal and one correction must round like an IEEE division."""
    M, K, group = 4096, 256, 32
    rng = np.random.default_rng(9)
    x = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-133, 127, size=(M, 1))).astype(np.float32)
    bits = f32_to_bf16_bits(x)
    for fmt in ("e4m3", "e2m1"):
        assert_bit_exact(Case(bits, K, group, fmt, "fp32", "row"))


# ----------------------------------------------------------- large index

def test_beyond_2_31_elements():
    """A matrix of more than 2^31 elements (64-bit addressing): sampled rows
    checked against the oracle.  The input tiles a 999-row host block so
    that a wrapped 32-bit offset would read a different row."""
    import torch
    block_rows, K, group = 999, 16512, 128
    M = (1 << 31) // K + 1000
    block = random_bf16(123, block_rows, K)
    dev_block = torch.from_numpy(block.view(np.int16)).cuda()
    x = torch.empty((M, K), dtype=torch.int16, device="cuda")
    for r0 in range(0, M, block_rows):
        n = min(block_rows, M - r0)
        x[r0:r0 + n] = dev_block[:n]
    codes = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    G = K // group
    scales = torch.empty((M, G), dtype=torch.float32, device="cuda")
    tk.tk_per_token_cast(x.data_ptr(), M, K, K, group, 0, 0, 0,
                         codes.data_ptr(), K, scales.data_ptr(), G,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    edge = (1 << 31) // K
    sample = sorted(set([0, 1, M // 2, edge - 1, edge, edge + 1, M - 2, M - 1] +
                        list(np.random.default_rng(1).integers(0, M, 40))))
    ref_c, ref_s = oracle.per_token_cast(block, K, group, oracle.FMT_E4M3,
                                         oracle.SCALE_FP32,
                                         oracle.LAYOUT_ROW_MAJOR,
                                         threads=THREADS)
    idx = torch.tensor(sample, device="cuda")
    got_c = codes.index_select(0, idx).cpu().numpy()
    got_s = scales.index_select(0, idx).cpu().numpy()
    for i, m in enumerate(sample):
        assert np.array_equal(got_c[i], ref_c[m % block_rows]), m
        assert np.array_equal(got_s[i].view(np.uint32),
                              ref_s[m % block_rows].view(np.uint32)), m
    del x, codes, scales
    torch.cuda.empty_cache()


# --------------------------------------------------------------- SwiGLU

@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["fp32", "pow2", "ue8m0"])
@pytest.mark.parametrize("layout", ["row", "transposed"])
def test_swiglu_small(fmt, mode, layout):
    for (M, N, group) in [(3, 128, 128), (254, 2048, 128), (37, 272, 16),
                          (5, 96, 32)]:
        bits = random_bf16(M * N + group, M, 2 * N, scale=2.0)
        case = Case(bits, N, group, fmt, mode, layout, swiglu=True)
        check_swiglu(case, max_code_frac=2e-3 if M * N < 5000 else 1e-4)


def test_swiglu_fp32_scales_track_the_exact_product():
    """fp32 scales of the fused path: every group's amax element re-evaluated
    to ~2^-44, so the scale equals the oracle's (correctly rounded product)
    except within ~2^-44 of a rounding midpoint.  Gates span [-80, 80],
    with a few beyond (the double-precision fallback)."""
    M, N, group = 512, 1024, 32
    rng = np.random.default_rng(21)
    gate = rng.uniform(-80, 80, size=(M, N)).astype(np.float32)
    gate[::7] = rng.standard_normal((gate[::7].shape)).astype(np.float32)
    up = (rng.standard_normal((M, N)) *
          10.0 ** rng.uniform(-3, 6, size=(M, 1))).astype(np.float32)
    # row 3: each group's amax element has |gate| > 80 (double fallback);
    # gate * up stays finite in fp32, as the contract requires
    gate[3] = rng.standard_normal(N).astype(np.float32) * 0.01
    up[3] = rng.standard_normal(N).astype(np.float32) * 0.01
    gate[3, [0, 32, 64, 96]] = [85.0, -90.0, -87.5, 90.0]
    up[3, [0, 32, 64, 96]] = [2.0, 3e36, 5e35, -3.0]
    bits = f32_to_bf16_bits(np.concatenate([gate, up], axis=1))
    case = Case(bits, N, group, "e4m3", "fp32", "row", swiglu=True)
    gc, gs = case.run_gpu()
    rc, rs = case.run_oracle()
    check_swiglu(case, gpu=(gc, gs), ref=(rc, rs), max_code_frac=2e-4)
    G = N // group
    sg = gs[1:-1, :G].view(np.int32).astype(np.int64)
    sr = rs[1:-1, :G].view(np.int32).astype(np.int64)
    assert np.count_nonzero(sg != sr) <= 2, np.count_nonzero(sg != sr)


def _near_edge_pairs(fmt_max, rng):
    """BF16 (gate, up) bit pairs whose SwiGLU value lies within a relative
    2^-13 of +-fmt_max * 2^j, where the power-of-two scale changes, and the
    relative offset of each.  Found by enumerating BF16 gates in [-6, 10]
    and ups of every mantissa over 22 binades with the plain double
    formula; this only chooses inputs (the expected values are the
    oracle's)."""
    g = np.arange(0, 0x10000, dtype=np.uint32)
    g = g[((g >> 7) & 0xFF) != 0xFF]                 # finite patterns only
    gv = bf16_bits_to_f32(g.astype(np.uint16)).astype(np.float64)
    gsel = g[(gv >= -6) & (gv <= 10) & (np.abs(gv) > 0.05)]
    ub = np.array([(e << 7) | m for e in range(114, 136) for m in range(128)],
                  np.uint32)
    gq = bf16_bits_to_f32(gsel.astype(np.uint16)).astype(np.float64)
    uq = bf16_bits_to_f32(ub.astype(np.uint16)).astype(np.float64)
    y = np.abs(gq[:, None] * uq[None, :] / (1.0 + np.exp(-gq[:, None])))
    t = np.log2(y / fmt_max)
    rel = (t - np.round(t)) * np.log(2.0)        # relative offset from the edge
    gi, ui = np.nonzero((np.abs(rel) <= 2.0 ** -13) & (y >= 1e-2))
    sign = rng.integers(0, 2, gi.size).astype(np.uint32) << 15
    return gsel[gi], ub[ui] | sign, rel[gi, ui]


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("mode", ["pow2", "ue8m0"])
def test_swiglu_pow2_scales_at_the_switching_points(fmt, mode):
    """Power-of-two scales where they change: every group's amax element
    sits within a relative 2^-13 of fmt_max * 2^j, about half of them
    inside the +-2^-15 band that the kernel re-evaluates exactly and the
    rest on the side it settles from the fp32 amax alone.  The scale bytes
    must equal the oracle's exactly (no edge allowance)."""
    fmt_max = 448.0 if fmt == "e4m3" else 6.0
    rng = np.random.default_rng(31)
    pg, pu, rel = _near_edge_pairs(fmt_max, rng)
    inner = np.abs(rel) <= 2.0 ** -15
    assert inner.sum() >= 200 and (~inner).sum() >= 200
    M, N, group = 64, 2048, 128
    G = N // group
    pick = rng.integers(0, pg.size, M * G)
    assert inner[pick].sum() >= 100 and (~inner[pick]).sum() >= 100
    gate = np.clip(rng.standard_normal((M, N)), -3, 3).astype(np.float32)
    up = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    gate_b = f32_to_bf16_bits(gate)
    up_b = f32_to_bf16_bits(up)
    ga = bf16_bits_to_f32(pg[pick].astype(np.uint16))
    ua = bf16_bits_to_f32(pu[pick].astype(np.uint16))
    y_edge = np.abs(ga.astype(np.float64) * ua / (1.0 + np.exp(-ga.astype(np.float64))))
    planted = np.empty((M, G), np.int64)
    for k in range(M * G):
        m, j = divmod(k, G)
        cols = slice(j * group, (j + 1) * group)
        # the others stay below 0.3 of the edge element: |silu(g)| <= 3
        up_b[m, cols] = f32_to_bf16_bits(up[m, cols] * np.float32(0.1 * y_edge[k]))
        at = j * group + int(rng.integers(0, group))
        gate_b[m, at] = pg[pick[k]]
        up_b[m, at] = pu[pick[k]]
        planted[m, j] = at
    bits = np.concatenate([gate_b, up_b], axis=1)
    # the planted element is its group's amax in the oracle's values
    y = np.abs(oracle.swiglu_values(bits, N, threads=THREADS)).reshape(M, G, group)
    assert np.array_equal(y.argmax(axis=2) + np.arange(G) * group, planted)
    case = Case(bits, N, group, fmt, mode, "row", swiglu=True)
    gc, gs = case.run_gpu()
    rc, rs = case.run_oracle()
    assert np.array_equal(gs, rs), np.count_nonzero(gs != rs)
    check_swiglu(case, gpu=(gc, gs), ref=(rc, rs), max_code_frac=2e-3)


def test_swiglu_zero_gate_and_strided():
    M, N, group = 33, 256, 64
    bits = random_bf16(8, M, 2 * N)
    bits[4, :N] = 0                              # gate 0 -> y 0 -> floor scale
    bits[5, N:] = 0                              # up 0 -> y 0
    case = Case(bits, N, group, "e4m3", "fp32", "row", swiglu=True,
                ld_x=2 * N + 40, code_pad=16, scale_pad=1)
    check_swiglu(case)


# -------------------------------------------------------- streams / API

def test_nondefault_stream_and_tensor_api():
    import torch
    M, K = 300, 1024
    bits = random_bf16(3, M, K)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        codes, scales = tk.per_token_cast(x, group=64, fmt="e4m3",
                                          scale="ue8m0", layout="transposed")
    s.synchronize()
    rc, rs = oracle.per_token_cast(bits, K, 64, oracle.FMT_E4M3,
                                   oracle.SCALE_UE8M0,
                                   oracle.LAYOUT_TRANSPOSED)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy()[:, :M], rs[:, :M])
    # host tensors in, host tensors out (copies inside the call)
    xh = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    hc, hs = tk.per_token_cast(xh, group=64, fmt="e4m3", scale="ue8m0",
                               layout="transposed")
    assert hc.device.type == "cpu"
    assert np.array_equal(hc.numpy(), rc)


@pytest.mark.parametrize("fmt,scale,layout,K,group", [
    ("e4m3", "ue8m0", "row", 7168, 128),
    ("e4m3", "fp32", "transposed", 1024, 32),
    ("e2m1", "ue8m0", "transposed", 272, 16),     # 136-byte code rows
    ("e2m1", "pow2", "row", 272, 16),
])
def test_host_buffers_match_device_path(fmt, scale, layout, K, group):
    """Host tensors in, host tensors out (copies inside the call): the
    results must equal the device-tensor call's bit for bit, including E2M1
    code rows whose device stride is padded to 16 bytes."""
    import torch
    M = 1613
    bits = random_bf16(21, M, K, scale=4.0)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    dc, ds = tk.per_token_cast(x.cuda(), group=group, fmt=fmt, scale=scale,
                               layout=layout)
    hc, hs = tk.per_token_cast(x.pin_memory(), group=group, fmt=fmt,
                               scale=scale, layout=layout)
    torch.cuda.synchronize()
    assert hc.device.type == "cpu" and hs.device.type == "cpu"
    assert np.array_equal(hc.numpy(), dc.cpu().numpy())
    if layout == "row":
        assert np.array_equal(hs.numpy().view(np.uint32),
                              ds.cpu().numpy().view(np.uint32))
    else:
        assert np.array_equal(hs.numpy().view(np.uint32)[:, :M],
                              ds.cpu().numpy().view(np.uint32)[:, :M])
    # the fused SwiGLU host path, same check
    bits2 = random_bf16(22, M, 2 * K)
    x2 = torch.from_numpy(bits2.view(np.int16)).view(torch.bfloat16)
    dc, ds = tk.swiglu_per_token_cast(x2.cuda(), group=group, fmt=fmt,
                                      scale=scale, layout=layout)
    hc, hs = tk.swiglu_per_token_cast(x2.pin_memory(), group=group, fmt=fmt,
                                      scale=scale, layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(hc.numpy(), dc.cpu().numpy())
    n = M if layout == "transposed" else None
    assert np.array_equal(hs.numpy().view(np.uint32)[..., :n],
                          ds.cpu().numpy().view(np.uint32)[..., :n])


@pytest.mark.parametrize("layout", ["row", "transposed"])
@pytest.mark.parametrize("chunk_rows", [4, 37, 0])
@pytest.mark.parametrize("swiglu", [False, True])
def test_host_entry_chunks_and_strides(layout, chunk_rows, swiglu):
    """The raw host-buffer entry: small and ragged chunks (37 rounds down to
    36), host row strides wider than the rows and not multiples of 16 (the
    input pad poisoned, the output pads filled with a sentinel that must
    survive), pageable numpy memory, and one stream listed twice.
    Results equal the device-tensor call's bit for bit."""
    import torch
    M, K, group, fmt, mode = 203, 384, 64, "e4m3", "fp32"
    in_cols = 2 * K if swiglu else K
    bits = random_bf16(41 + swiglu, M, in_cols, scale=3.0)
    ld_x = in_cols + 40
    xh = np.full((M, ld_x), 0x7FC0, np.uint16)            # NaN in the pad
    xh[:, :in_cols] = bits
    G = K // group
    ld_codes = K + 24
    codes = np.full((M, ld_codes), 0xA5, np.uint8)
    if layout == "row":
        ld_scales, scale_rows = G + 3, M
    else:
        ld_scales, scale_rows = M + 5, G
    scales = np.full((scale_rows, ld_scales), 0x7F7F7F7F, np.uint32)
    need = tk.tk_host_scratch_bytes(M, K, group, tk.FMT[fmt], tk.SCALE[mode],
                                    tk.LAYOUT[layout], int(swiglu))
    scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    entry = (tk.tk_swiglu_per_token_cast_host if swiglu
             else tk.tk_per_token_cast_host)
    entry(xh.ctypes.data, M, K, ld_x, group, tk.FMT[fmt], tk.SCALE[mode],
          tk.LAYOUT[layout], codes.ctypes.data, ld_codes, scales.ctypes.data,
          ld_scales, scratch.data_ptr(), need, chunk_rows, (s, s))
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    fn = tk.swiglu_per_token_cast if swiglu else tk.per_token_cast
    dc, ds = fn(x, group=group, fmt=fmt, scale=mode, layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(codes[:, :K], dc.cpu().numpy())
    assert (codes[:, K:] == 0xA5).all()
    want = ds.cpu().numpy().view(np.uint32)
    if layout == "row":
        assert np.array_equal(scales[:, :G], want[:, :G])
        assert (scales[:, G:] == 0x7F7F7F7F).all()
    else:
        assert np.array_equal(scales[:, :M], want[:, :M])
        assert (scales[:, M:] == 0x7F7F7F7F).all()


def test_bf16_input_values_roundtrip():
    """Sanity: the decoded codes times the scales approximate the input."""
    import torch
    bits = random_bf16(4, 64, 1024)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    codes, scales = tk.per_token_cast(x, group=128, fmt="e4m3", scale="fp32")
    deq = codes.view(torch.float8_e4m3fn).float().cpu().numpy() * \
        np.repeat(scales.cpu().numpy(), 128, axis=1)
    xf = bf16_bits_to_f32(bits)
    assert np.max(np.abs(deq - xf)) <= np.max(np.abs(xf)) / 16


def test_zz_no_kernel_gave_up_on_a_wait():
    """No kernel of this module's runs hit its bounded-wait limit."""
    assert tk.tk_get_device_fault(clear=True) == 0
