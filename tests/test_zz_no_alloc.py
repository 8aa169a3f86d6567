"""The allocation-free per-channel entry point against the workspace one
(GPU).

tk_per_channel_cast_noalloc keeps its workspace in the library's static
device memory and sets it up (address lookup, one clearing memset) on its
first call for a device.  This file is collected last on purpose, and its
tests pass both alone and after every other test: nothing here depends on
whether the set-up already happened.
"""
import numpy as np
import pytest

import precision_quantization_token_gb300 as tk
from precision_quantization_token_gb300.inputs import (WORKLOADS, make_input,
                                                       random_bf16)

pytestmark = pytest.mark.gpu

OPTIONS = [("e4m3", "fp32"), ("e4m3", "ue8m0"), ("e2m1", "pow2"),
           ("e2m1", "ue8m0")]


def _buffers(torch, M, K, fmt, mode):
    rb = K if fmt == "e4m3" else K // 2
    ld = (rb + 15) // 16 * 16
    codes = torch.full((M, ld), 0xA5, dtype=torch.uint8, device="cuda")
    nw = (K + 3) // 4 if mode == "ue8m0" else K
    scales = torch.full((nw + 8,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    return codes, ld, scales


def _launch(torch, entry, bits, fmt, mode):
    """Enqueue one cast on the current stream; returns its output tensors."""
    M, K = bits.shape
    x = torch.from_numpy(bits.view(np.int16)).cuda()
    codes, ld, scales = _buffers(torch, M, K, fmt, mode)
    stream = torch.cuda.current_stream().cuda_stream
    if entry == "noalloc":
        tk.tk_per_channel_cast_noalloc(x.data_ptr(), M, K, K, tk.FMT[fmt],
                                       tk.SCALE[mode], codes.data_ptr(), ld,
                                       scales.data_ptr() + 16, stream)
    else:
        ws = torch.zeros(tk.tk_per_channel_workspace_bytes(K),
                         dtype=torch.uint8, device="cuda")
        tk.tk_per_channel_cast(x.data_ptr(), M, K, K, tk.FMT[fmt],
                               tk.SCALE[mode], codes.data_ptr(), ld,
                               scales.data_ptr() + 16, ws.data_ptr(),
                               ws.numel(), stream)
    return x, codes, scales


def _host(out):
    _, codes, scales = out
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("fmt,mode", OPTIONS)
def test_two_calls_in_a_row_match_the_workspace_entry(fmt, mode):
    """Two allocation-free calls enqueued back to back (no sync between
    them), with different shapes and value ranges: the second must not see
    the first's column maxima; both equal the workspace entry's results."""
    import torch
    a = random_bf16(31, 700, 4096, scale=50.0)
    b = random_bf16(32, 300, 2064, scale=0.01)
    first = _launch(torch, "noalloc", a, fmt, mode)
    second = _launch(torch, "noalloc", b, fmt, mode)
    torch.cuda.synchronize()
    got = [_host(first), _host(second)]
    for bits, (gc, gs) in zip((a, b), got):
        ref = _launch(torch, "workspace", bits, fmt, mode)
        torch.cuda.synchronize()
        rc, rs = _host(ref)
        assert np.array_equal(gc, rc), "codes differ"
        assert np.array_equal(gs, rs), "scales differ"


def test_full_size_and_channel_limit():
    import torch
    bits = make_input(WORKLOADS["pc2"])
    got = _host(_launch(torch, "noalloc", bits, "e4m3", "fp32"))
    ref = _host(_launch(torch, "workspace", bits, "e4m3", "fp32"))
    torch.cuda.synchronize()
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    wide = random_bf16(33, 40, 65536)             # the largest K it takes
    got = _host(_launch(torch, "noalloc", wide, "e4m3", "ue8m0"))
    ref = _host(_launch(torch, "workspace", wide, "e4m3", "ue8m0"))
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    with pytest.raises(tk.TkError) as e:
        _launch(torch, "noalloc", random_bf16(34, 4, 65536 + 16), "e4m3",
                "fp32")
    assert e.value.status == 2                    # TK_ERR_UNSUPPORTED
    assert tk.tk_get_device_fault(clear=False) == 0
