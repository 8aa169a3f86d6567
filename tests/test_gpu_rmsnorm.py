"""RMSNorm fused with the per-token cast against the oracle (GPU).

The kernel computes RMSNorm in fp32 (one fixed summation order, IEEE steps)
and the oracle in double rounded once, so the compare is a tolerance one
(tests/gpu_util.check_close).  SCALE_ULPS follows from the kernel's
arithmetic: a lane keeps two sums of at most 24 squares each (23 roundings),
adds them (1), the warp tree adds 5 more and the group 5 more, then the
product by RN(1/K) (2 with the rounding of 1/K) and the addition of eps (1):
at most 37 ulps on the mean square; rsqrtf halves that and adds its own
error (at most 2 ulps), and the product by rstd one more: about 22 ulps
between the kernel's y and exact y, and one more for the oracle's rounding;
40 leaves room.  So:
  * fp32 scales within SCALE_ULPS ulps; UE8M0 / power-of-two scales equal
    except within SCALE_ULPS ulps of a power of two;
  * a code may differ only by one step, and only where the oracle's y / s
    lies within BAND_ULPS = 2 * SCALE_ULPS + 2 ulps of the midpoint between
    the two codes (y and s each off by at most SCALE_ULPS, plus the two
    quotients' roundings).  Such codes are not rare: x * w has 16
    significant bits and rstd cancels between y and s, so the exact
    quotient 448 * (x w) / max|x w| often falls on a midpoint exactly, and
    then rounding noise decides;
  * at most MAX_CODE_FRAC of the codes differ.
The tests print the largest deviations seen.
"""
import numpy as np
import pytest

import precision_quantization_token_gb300 as tk
from gpu_util import Case, check_close, torch_mod
from precision_quantization_token_gb300.inputs import (WORKLOADS, make_gain,
                                                       make_input, random_bf16)

pytestmark = pytest.mark.gpu

SCALE_ULPS = 40
BAND_ULPS = 2 * SCALE_ULPS + 2
MAX_CODE_FRAC = 1e-3
FMTS = ["e4m3", "e2m1"]
MODES = ["fp32", "pow2", "ue8m0"]


def gain(K, seed):
    rng = np.random.default_rng(seed)
    g = (1.0 + 0.1 * rng.standard_normal(K)).astype(np.float32)
    return (g.view(np.uint32) >> 16).astype(np.uint16)


def check(case):
    info = check_close(case, max_code_frac=MAX_CODE_FRAC, scale_ulps=SCALE_ULPS,
                       edge_ulps=SCALE_ULPS, band_ulps=BAND_ULPS)
    print(info)
    return info


def test_full_workload():
    w = WORKLOADS["r2"]
    case = Case(make_input(w), w.K, w.group, w.fmt, w.scale, w.layout,
                gain=make_gain(w), eps=w.eps)
    check(case)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("layout", ["row", "transposed"])
def test_every_option(fmt, mode, layout):
    bits = make_input(WORKLOADS["c2"], M=1024)
    for group in (16, 128):
        check(Case(bits, 7168, group, fmt, mode, layout, gain=gain(7168, 1),
                   eps=1e-6))


@pytest.mark.parametrize("M,K", [(1, 16), (3, 48), (257, 1040), (64, 6160),
                                 (200, 8192), (5, 4096)])
def test_shapes(M, K):
    bits = random_bf16(M * 3 + K, M, K, scale=2.0)
    for fmt, mode in (("e4m3", "fp32"), ("e2m1", "ue8m0")):
        check(Case(bits, K, 16, fmt, mode, "row", gain=gain(K, K), eps=1e-5))


def test_strides_and_pads():
    bits = random_bf16(5, 300, 2048)
    case = Case(bits, 2048, 64, "e4m3", "fp32", "transposed", ld_x=2104,
                code_pad=48, scale_pad=2, gain=gain(2048, 2), eps=1e-6)
    check(case)
    case = Case(bits, 2048, 32, "e2m1", "ue8m0", "row", ld_x=2056,
                code_pad=16, scale_pad=3, gain=gain(2048, 3), eps=1e-6)
    check(case)


def test_value_extremes():
    """Rows spread over magnitudes, zero rows (eps > 0: y = +-0), rows of
    BF16 denormals (eps dominates), a lone outlier per row, and a gain with
    zeros and negative values."""
    M, K = 96, 1024
    rng = np.random.default_rng(9)
    v = rng.standard_normal((M, K)).astype(np.float32)
    v *= np.exp2(rng.integers(-30, 31, (M, 1))).astype(np.float32)
    bits = (v.view(np.uint32) >> 16).astype(np.uint16)
    bits[10] = 0
    bits[11] = 0x8000
    bits[12] = (rng.integers(1, 128, K) | (rng.integers(0, 2, K) << 15)).astype(np.uint16)
    bits[13, :] = 0x3C00                                   # 1/128 everywhere ...
    bits[13, 77] = 0x4700                                  # ... and one 32768
    g = gain(K, 4)
    g[::17] = 0
    g[5::29] |= 0x8000
    for eps in (1e-6, 0.5):
        for fmt, mode in (("e4m3", "fp32"), ("e4m3", "ue8m0"), ("e2m1", "pow2")):
            check(Case(bits, K, 128, fmt, mode, "row", gain=g, eps=eps))


def test_eps_zero_on_nonzero_rows():
    bits = random_bf16(6, 128, 512)
    check(Case(bits, 512, 128, "e4m3", "fp32", "row", gain=gain(512, 6),
               eps=0.0))


def test_tensor_api():
    torch = torch_mod()
    import oracle
    bits = random_bf16(7, 64, 1024)
    g = gain(1024, 7)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    w = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).cuda()
    codes, scales = tk.rmsnorm_per_token_cast(x, w, eps=1e-6, group=128,
                                              fmt="e4m3", scale="ue8m0")
    rc, rs = oracle.rmsnorm_per_token_cast(bits, g, 1024, 1e-6, 128,
                                           oracle.FMT_E4M3, oracle.SCALE_UE8M0,
                                           oracle.LAYOUT_ROW_MAJOR)
    gc = codes.cpu().numpy()
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert (gc != rc).mean() <= 1e-3



def test_beyond_2_31_elements():
    """More than 2^31 elements: the input repeats a 997-row host block, so
    row m equals host row m % 997; sampled rows on both sides of 2^31
    elements must equal the kernel's own result for those host rows (a
    small launch) exactly, and that result meets the tolerance above."""
    import oracle
    torch = torch_mod()
    K, hb, group = 8192, 997, 128
    M = (1 << 31) // K + 1000
    block = random_bf16(126, hb, K, scale=2.0)
    g = gain(K, 126)
    small = Case(block, K, group, "e4m3", "ue8m0", "row", gain=g, eps=1e-6)
    check(small)                                   # the host rows themselves
    ref_codes, ref_scales = small.run_gpu()
    dev_block = torch.from_numpy(block.view(np.int16)).cuda()
    x = torch.empty((M, K), dtype=torch.int16, device="cuda")
    for r0 in range(0, M, hb):
        n = min(hb, M - r0)
        x[r0:r0 + n] = dev_block[:n]
    wd = torch.from_numpy(g.view(np.int16)).cuda()
    codes = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    G = K // group
    scales = torch.empty((M, (G + 3) // 4), dtype=torch.int32, device="cuda")
    tk.tk_rmsnorm_per_token_cast(x.data_ptr(), wd.data_ptr(), M, K, K, 1e-6,
                                 group, tk.FMT["e4m3"], tk.SCALE["ue8m0"],
                                 tk.LAYOUT["row"], codes.data_ptr(), K,
                                 scales.data_ptr(), scales.shape[1],
                                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    edge = (1 << 31) // K
    sample = sorted({0, 1, M // 2, edge - 1, edge, edge + 1, M - 2, M - 1})
    idx = torch.tensor(sample, device="cuda")
    got_c = codes.index_select(0, idx).cpu().numpy()
    got_s = scales.index_select(0, idx).cpu().numpy().view(np.uint32)
    for i, m in enumerate(sample):
        assert np.array_equal(got_c[i], ref_codes[1 + m % hb, :K]), m
        assert np.array_equal(got_s[i], ref_scales[1 + m % hb, :(G + 3) // 4]), m
    del x, codes, scales
    torch.cuda.empty_cache()


def test_zz_no_kernel_gave_up_on_a_wait():
    assert tk.tk_get_device_fault(clear=False) == 0
