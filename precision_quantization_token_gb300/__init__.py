"""GB300-native per-token group-wise activation cast (BF16 -> FP8 E4M3 / FP4 E2M1).

Thin Python binding over the C-ABI library built from ``csrc/`` (declared in
``include/tk_cast.h``).  The binding only marshals arguments: PyTorch provides
device memory and the current stream, and every step of the cast runs in the
library's CUDA kernel.  There is no CPU fallback: if the library is missing,
every call raises.

Low level (same names and arguments as the C ABI, raw pointers and sizes):
    tk_per_token_cast(x_ptr, M, K, ld_x, group, fmt, mode, layout,
                      codes_ptr, ld_codes, scales_ptr, ld_scales, stream)
    tk_swiglu_per_token_cast(x_ptr, M, N, ld_x, ...)
    tk_per_token_dequant(codes_ptr, ld_codes, scales_ptr, ld_scales, M, K,
                         group, fmt, mode, layout, y_ptr, ld_y, out_dtype, stream)
    tk_per_token_cast_back(x_ptr, M, K, ld_x, group, fmt, mode, y_ptr, ld_y,
                           stream)
    tk_rmsnorm_per_token_cast(x_ptr, w_ptr, M, K, ld_x, eps, group, fmt,
                              mode, layout, codes_ptr, ld_codes, scales_ptr,
                              ld_scales, stream)
    tk_per_block_cast(x_ptr, M, K, ld_x, fmt, mode, codes_ptr, ld_codes,
                      scales_ptr, ld_scales, stream)
    tk_per_channel_cast(x_ptr, M, K, ld_x, fmt, mode, codes_ptr, ld_codes,
                        scales_ptr, workspace_ptr, workspace_bytes, stream)
    tk_per_channel_workspace_bytes(K)
    tk_per_block_dequant(codes_ptr, ld_codes, scales_ptr, ld_scales, M, K,
                         fmt, mode, y_ptr, ld_y, out_dtype, stream)
    tk_per_channel_dequant(codes_ptr, ld_codes, scales_ptr, M, K, fmt, mode,
                           y_ptr, ld_y, out_dtype, stream)
    tk_per_channel_cast_noalloc(x_ptr, M, K, ld_x, fmt, mode, codes_ptr,
                                ld_codes, scales_ptr, stream)

Tensor level (allocates outputs with torch):
    codes, scales = per_token_cast(x, group=128, fmt="e4m3", scale="fp32",
                                   layout="row")
    codes, scales = swiglu_per_token_cast(x, group=128, ...)  # x = [gate|up]
    y = per_token_dequant(codes, scales, K, group=128, fmt="e4m3", ...)
    y = per_token_cast_back(x, group=128, fmt="e4m3", scale="fp32")
    codes, scales = rmsnorm_per_token_cast(x, w, eps=1e-6, group=128, ...)
    codes, scales = per_block_cast(x, fmt="e4m3", scale="fp32")   # 128x128
    codes, scales = per_channel_cast(x, fmt="e4m3", scale="fp32")
    y = per_block_dequant(codes, scales, K, fmt="e4m3", scale="fp32")
    y = per_channel_dequant(codes, scales, K, fmt="e4m3", scale="fp32")

Operation (TileKernels README, "Features"; aiwiki "TileKernels", section
"Quantization"): per row and per group of 16/32/64/128 channels, amax, a
scale max(amax, 1e-4)/fmt_max (fp32, or rounded up to 2^k, optionally packed
as UE8M0 bytes four per int32), and round-to-nearest-even saturated codes;
scales row-major or transposed with M padded ("DeepGEMM's layout").
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

FMT = {"e4m3": 0, "e2m1": 1}
OUT_DTYPE = {"bf16": 0, "fp32": 1}
SCALE = {"fp32": 0, "pow2": 1, "ue8m0": 2}
LAYOUT = {"row": 0, "transposed": 1}

TK_OK = 0
STATUS_NAMES = {0: "TK_OK", 1: "TK_ERR_INVALID_ARG", 2: "TK_ERR_UNSUPPORTED",
                3: "TK_ERR_MISALIGNED", 4: "TK_ERR_CUDA"}

_lib = None
_lock = threading.Lock()


class TkError(RuntimeError):
    """A non-OK status returned by the library."""

    def __init__(self, status: int, detail: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, f"status {status}")
        super().__init__(f"{name}{': ' + detail if detail else ''}")


def library_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in-tree)."""
    return _build.build(force=force)


def load():
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library not built ({path} missing); run "
                    "precision_quantization_token_gb300.build() first")
            lib = ctypes.CDLL(path)
            i64, p, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            sig = [p, i64, i64, i64, i, i, i, i, p, i64, p, i64, p]
            for name in ("tk_per_token_cast", "tk_swiglu_per_token_cast"):
                fn = getattr(lib, name)
                fn.argtypes = sig
                fn.restype = i
            lib.tk_per_token_cast_back.argtypes = [p, i64, i64, i64, i, i, i,
                                                   p, i64, p]
            lib.tk_per_token_cast_back.restype = i
            lib.tk_per_token_dequant.argtypes = [p, i64, p, i64, i64, i64, i, i,
                                                 i, i, p, i64, i, p]
            lib.tk_per_token_dequant.restype = i
            lib.tk_rmsnorm_per_token_cast.argtypes = [p, p, i64, i64, i64,
                                                      ctypes.c_float, i, i, i,
                                                      i, p, i64, p, i64, p]
            lib.tk_rmsnorm_per_token_cast.restype = i
            lib.tk_per_block_cast.argtypes = [p, i64, i64, i64, i, i, p, i64,
                                              p, i64, p]
            lib.tk_per_block_cast.restype = i
            lib.tk_per_channel_cast.argtypes = [p, i64, i64, i64, i, i, p, i64,
                                                p, p, ctypes.c_size_t, p]
            lib.tk_per_channel_cast.restype = i
            lib.tk_per_channel_cast_noalloc.argtypes = [p, i64, i64, i64, i, i,
                                                        p, i64, p, p]
            lib.tk_per_channel_cast_noalloc.restype = i
            lib.tk_per_block_dequant.argtypes = [p, i64, p, i64, i64, i64, i,
                                                 i, p, i64, i, p]
            lib.tk_per_block_dequant.restype = i
            lib.tk_per_channel_dequant.argtypes = [p, i64, p, i64, i64, i, i,
                                                   p, i64, i, p]
            lib.tk_per_channel_dequant.restype = i
            lib.tk_per_channel_workspace_bytes.argtypes = [i64]
            lib.tk_per_channel_workspace_bytes.restype = ctypes.c_size_t
            lib.tk_host_scratch_bytes.argtypes = [i64, i64, i, i, i, i, i]
            lib.tk_host_scratch_bytes.restype = ctypes.c_size_t
            hsig = [p, i64, i64, i64, i, i, i, i, p, i64, p, i64, p,
                    ctypes.c_size_t, i64, ctypes.POINTER(p), i]
            for name in ("tk_per_token_cast_host",
                         "tk_swiglu_per_token_cast_host"):
                fn = getattr(lib, name)
                fn.argtypes = hsig
                fn.restype = i
            lib.tk_get_device_fault.argtypes = [p, i]
            lib.tk_get_device_fault.restype = i
            lib.tk_status_string.argtypes = [i]
            lib.tk_status_string.restype = ctypes.c_char_p
            lib.tk_last_cuda_error.argtypes = []
            lib.tk_last_cuda_error.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _check(status: int):
    if status != TK_OK:
        detail = ""
        if status == 4:
            detail = load().tk_last_cuda_error().decode()
        raise TkError(status, detail)


# ------------------------------------------------------------- C-ABI names

def tk_per_token_cast(x_ptr, M, K, ld_x, group, fmt, mode, layout, codes_ptr,
                      ld_codes, scales_ptr, ld_scales, stream=0) -> None:
    """Raw-pointer call of the C entry point; raises TkError on failure."""
    _check(load().tk_per_token_cast(x_ptr, M, K, ld_x, group, fmt, mode,
                                    layout, codes_ptr, ld_codes, scales_ptr,
                                    ld_scales, stream))


def tk_swiglu_per_token_cast(x_ptr, M, N, ld_x, group, fmt, mode, layout,
                             codes_ptr, ld_codes, scales_ptr, ld_scales,
                             stream=0) -> None:
    """Raw-pointer call of the fused SwiGLU entry point."""
    _check(load().tk_swiglu_per_token_cast(x_ptr, M, N, ld_x, group, fmt,
                                           mode, layout, codes_ptr, ld_codes,
                                           scales_ptr, ld_scales, stream))


def tk_per_token_cast_back(x_ptr, M, K, ld_x, group, fmt, mode, y_ptr, ld_y,
                           stream=0) -> None:
    """Raw-pointer call of the cast-and-cast-back entry point."""
    _check(load().tk_per_token_cast_back(x_ptr, M, K, ld_x, group, fmt, mode,
                                         y_ptr, ld_y, stream))


def tk_per_token_dequant(codes_ptr, ld_codes, scales_ptr, ld_scales, M, K,
                         group, fmt, mode, layout, y_ptr, ld_y, out_dtype,
                         stream=0) -> None:
    """Raw-pointer call of the dequantization entry point."""
    _check(load().tk_per_token_dequant(codes_ptr, ld_codes, scales_ptr,
                                       ld_scales, M, K, group, fmt, mode,
                                       layout, y_ptr, ld_y, out_dtype, stream))


def tk_rmsnorm_per_token_cast(x_ptr, w_ptr, M, K, ld_x, eps, group, fmt,
                              mode, layout, codes_ptr, ld_codes, scales_ptr,
                              ld_scales, stream=0) -> None:
    """Raw-pointer call of RMSNorm (gain w, eps) fused with the per-token
    cast of its output."""
    _check(load().tk_rmsnorm_per_token_cast(x_ptr, w_ptr, M, K, ld_x, eps,
                                            group, fmt, mode, layout,
                                            codes_ptr, ld_codes, scales_ptr,
                                            ld_scales, stream))


def tk_per_block_cast(x_ptr, M, K, ld_x, fmt, mode, codes_ptr, ld_codes,
                      scales_ptr, ld_scales, stream=0) -> None:
    """Raw-pointer call of the per-block (128 x 128) cast."""
    _check(load().tk_per_block_cast(x_ptr, M, K, ld_x, fmt, mode, codes_ptr,
                                    ld_codes, scales_ptr, ld_scales, stream))


def tk_per_channel_cast(x_ptr, M, K, ld_x, fmt, mode, codes_ptr, ld_codes,
                        scales_ptr, workspace_ptr, workspace_bytes,
                        stream=0) -> None:
    """Raw-pointer call of the per-channel cast (caller's workspace)."""
    _check(load().tk_per_channel_cast(x_ptr, M, K, ld_x, fmt, mode, codes_ptr,
                                      ld_codes, scales_ptr, workspace_ptr,
                                      workspace_bytes, stream))


def tk_per_channel_cast_noalloc(x_ptr, M, K, ld_x, fmt, mode, codes_ptr,
                                ld_codes, scales_ptr, stream=0) -> None:
    """Raw-pointer call of the per-channel cast on the library's static
    per-device workspace (K <= 65536; calls must not overlap in time)."""
    _check(load().tk_per_channel_cast_noalloc(x_ptr, M, K, ld_x, fmt, mode,
                                              codes_ptr, ld_codes, scales_ptr,
                                              stream))


def tk_per_block_dequant(codes_ptr, ld_codes, scales_ptr, ld_scales, M, K,
                         fmt, mode, y_ptr, ld_y, out_dtype, stream=0) -> None:
    """Raw-pointer call of the per-block dequantization."""
    _check(load().tk_per_block_dequant(codes_ptr, ld_codes, scales_ptr,
                                       ld_scales, M, K, fmt, mode, y_ptr,
                                       ld_y, out_dtype, stream))


def tk_per_channel_dequant(codes_ptr, ld_codes, scales_ptr, M, K, fmt, mode,
                           y_ptr, ld_y, out_dtype, stream=0) -> None:
    """Raw-pointer call of the per-channel dequantization."""
    _check(load().tk_per_channel_dequant(codes_ptr, ld_codes, scales_ptr, M,
                                         K, fmt, mode, y_ptr, ld_y, out_dtype,
                                         stream))


def tk_per_channel_workspace_bytes(K: int) -> int:
    return int(load().tk_per_channel_workspace_bytes(K))


def tk_host_scratch_bytes(M, K, group, fmt, mode, layout, swiglu=0) -> int:
    """Device scratch bytes of the host-buffer casts (0: bad arguments)."""
    return int(load().tk_host_scratch_bytes(M, K, group, fmt, mode, layout,
                                            swiglu))


def _stream_array(streams):
    arr = (ctypes.c_void_p * len(streams))(*[s or None for s in streams])
    return arr, len(streams)


def tk_per_token_cast_host(x_ptr, M, K, ld_x, group, fmt, mode, layout,
                           codes_ptr, ld_codes, scales_ptr, ld_scales,
                           scratch_ptr, scratch_bytes, chunk_rows=0,
                           streams=(0,)) -> None:
    """Raw-pointer call of the host-buffer cast (host x, codes, scales;
    device scratch; chunks dealt over the cudaStream_t handles in
    `streams`); blocks until the outputs are in host memory."""
    arr, n = _stream_array(streams)
    _check(load().tk_per_token_cast_host(x_ptr, M, K, ld_x, group, fmt, mode,
                                         layout, codes_ptr, ld_codes,
                                         scales_ptr, ld_scales, scratch_ptr,
                                         scratch_bytes, chunk_rows, arr, n))


def tk_swiglu_per_token_cast_host(x_ptr, M, N, ld_x, group, fmt, mode, layout,
                                  codes_ptr, ld_codes, scales_ptr, ld_scales,
                                  scratch_ptr, scratch_bytes, chunk_rows=0,
                                  streams=(0,)) -> None:
    """Raw-pointer call of the host-buffer fused SwiGLU cast."""
    arr, n = _stream_array(streams)
    _check(load().tk_swiglu_per_token_cast_host(
        x_ptr, M, N, ld_x, group, fmt, mode, layout, codes_ptr, ld_codes,
        scales_ptr, ld_scales, scratch_ptr, scratch_bytes, chunk_rows, arr,
        n))


def tk_get_device_fault(clear: bool = False) -> int:
    """The device fault word of the current device (0: no kernel gave up on
    a wait); see include/tk_cast.h."""
    word = ctypes.c_uint(0)
    _check(load().tk_get_device_fault(ctypes.byref(word), int(clear)))
    return word.value


def tk_status_string(status: int) -> str:
    return load().tk_status_string(status).decode()


# ---------------------------------------------------------- tensor helpers

def scale_shape(M: int, K: int, group: int, scale: str = "fp32",
                layout: str = "row", m_pad_to: int = 4):
    """Shape and torch dtype name of the scale tensor for an [M, K] cast."""
    G = K // group
    words = (G + 3) // 4 if scale == "ue8m0" else G
    dtype = "int32" if scale == "ue8m0" else "float32"
    if layout == "row":
        return (M, words), dtype
    m_pad = (M + m_pad_to - 1) // m_pad_to * m_pad_to
    return (words, m_pad), dtype


def _code_buffer(torch, M, K, fmt, device):
    """uint8 [M, K or K/2] codes whose rows start on 16-byte boundaries (a
    view of a buffer with the row stride rounded up to 16 bytes)."""
    row_bytes = K if fmt == "e4m3" else K // 2
    ld = (row_bytes + 15) // 16 * 16
    return torch.empty((M, ld), dtype=torch.uint8, device=device)[:, :row_bytes]


def _outputs(torch, M, K, group, fmt, scale, layout, device, codes, scales):
    if codes is None:
        codes = _code_buffer(torch, M, K, fmt, device)
    if scales is None:
        shape, dt = scale_shape(M, K, group, scale, layout)
        scales = torch.empty(shape, dtype=getattr(torch, dt), device=device)
    return codes, scales


_host_streams = {}
_host_scratch = {}
_host_lock = threading.Lock()


HOST_STREAMS = 4    # streams the host-buffer pipeline deals its chunks over


def _copy_streams(torch, device):
    """The host-buffer pipeline's streams for a device (created once), and
    their handles as a ctypes array."""
    key = torch.device(device).index
    if key not in _host_streams:
        streams = tuple(torch.cuda.Stream(device) for _ in range(HOST_STREAMS))
        _host_streams[key] = (streams,
                              _stream_array([st.cuda_stream for st in streams]))
    return _host_streams[key]


def _call(entry, x, K, group, fmt, scale, layout, codes, scales, stream):
    import torch
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bfloat16 tensor with unit column "
                         "stride")
    if x.device.type == "cpu":
        return _call_host(entry, torch, x, K, group, fmt, scale, layout,
                          codes, scales)
    M = x.shape[0]
    codes, scales = _outputs(torch, M, K, group, fmt, scale, layout, x.device,
                             codes, scales)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    entry(x.data_ptr(), M, K, x.stride(0), group, FMT[fmt], SCALE[scale],
          LAYOUT[layout], codes.data_ptr(), codes.stride(0),
          scales.data_ptr(), scales.stride(0), stream)
    return codes, scales


def _call_host(entry, torch, x, K, group, fmt, scale, layout, codes, scales):
    """CPU tensors: the library's host-buffer pipeline (chunks of rows
    uploaded, cast and downloaded on HOST_STREAMS streams) on the current
    device."""
    M = x.shape[0]
    swiglu = entry is tk_swiglu_per_token_cast
    if codes is None:
        row_bytes = K if fmt == "e4m3" else K // 2
        codes = torch.empty((M, row_bytes), dtype=torch.uint8, pin_memory=True)
    if scales is None:
        shape, dt = scale_shape(M, K, group, scale, layout)
        scales = torch.empty(shape, dtype=getattr(torch, dt), pin_memory=True)
    if codes.device.type != "cpu" or scales.device.type != "cpu":
        raise ValueError("a CPU input takes CPU codes and scales")
    device = torch.device("cuda", torch.cuda.current_device())
    need = tk_host_scratch_bytes(M, K, group, FMT[fmt], SCALE[scale],
                                 LAYOUT[layout], int(swiglu))
    host_entry = (load().tk_swiglu_per_token_cast_host if swiglu
                  else load().tk_per_token_cast_host)
    # One scratch per device, grown on demand and reused: the call returns
    # only after every stream it used is idle, and the lock keeps two host
    # threads from sharing it (or the streams) at once.
    with _host_lock:
        streams, (arr, n) = _copy_streams(torch, device)
        scratch = _host_scratch.get(device.index)
        if scratch is None or scratch.numel() < need:
            torch.cuda.synchronize(device)
            _host_scratch.pop(device.index, None)
            with torch.cuda.stream(streams[0]):
                scratch = torch.empty(max(need, 16), dtype=torch.uint8,
                                      device=device)
            _host_scratch[device.index] = scratch
        _check(host_entry(x.data_ptr(), M, K, x.stride(0), group, FMT[fmt],
                          SCALE[scale], LAYOUT[layout], codes.data_ptr(),
                          codes.stride(0), scales.data_ptr(),
                          scales.stride(0), scratch.data_ptr(), need, 0, arr,
                          n))
    return codes, scales


def per_token_cast(x, group: int = 128, fmt: str = "e4m3",
                   scale: str = "fp32", layout: str = "row", *, codes=None,
                   scales=None, stream=None):
    """Per-token group-wise cast of a bfloat16 [M, K] tensor.

    CUDA input: outputs are CUDA tensors, the call is asynchronous on the
    current stream.  CPU input (preferably pinned): the library's host-buffer
    pipeline uploads the rows in chunks to the current CUDA device, casts
    them there and downloads codes and scales into (pinned) host tensors,
    chunks dealt over HOST_STREAMS streams; returns once they are on the
    host.  The device scratch it stages through (the largest needed so
    far) is kept per device for later calls.
    Returns (codes uint8 [M, K or K/2], scales) -- see ``scale_shape``.
    """
    K = x.shape[1]
    return _call(tk_per_token_cast, x, K, group, fmt, scale, layout, codes,
                 scales, stream)


def swiglu_per_token_cast(x, group: int = 128, fmt: str = "e4m3",
                          scale: str = "fp32", layout: str = "row", *,
                          codes=None, scales=None, stream=None):
    """Fused SwiGLU + per-token cast of x = [gate | up] (bfloat16 [M, 2N])."""
    if x.shape[1] % 2:
        raise ValueError("x must hold [gate | up] halves of equal width")
    N = x.shape[1] // 2
    return _call(tk_swiglu_per_token_cast, x, N, group, fmt, scale, layout,
                 codes, scales, stream)


def rmsnorm_per_token_cast(x, w, eps: float = 1e-6, group: int = 128,
                           fmt: str = "e4m3", scale: str = "fp32",
                           layout: str = "row", *, codes=None, scales=None,
                           stream=None):
    """RMSNorm of the rows of a bfloat16 [M, K] CUDA tensor with gain w
    (bfloat16 [K]) fused with the per-token cast of the fp32 result.
    Returns (codes, scales) as per_token_cast does."""
    import torch
    _check_x(x)
    if w.dtype != torch.bfloat16 or w.dim() != 1 or w.stride(0) != 1:
        raise ValueError("w must be a contiguous 1-D bfloat16 tensor")
    M, K = x.shape
    codes, scales = _outputs(torch, M, K, group, fmt, scale, layout, x.device,
                             codes, scales)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    tk_rmsnorm_per_token_cast(x.data_ptr(), w.data_ptr(), M, K, x.stride(0),
                              eps, group, FMT[fmt], SCALE[scale],
                              LAYOUT[layout], codes.data_ptr(),
                              codes.stride(0), scales.data_ptr(),
                              scales.stride(0), stream)
    return codes, scales


def per_token_dequant(codes, scales, K: int, group: int = 128,
                      fmt: str = "e4m3", scale: str = "fp32",
                      layout: str = "row", out_dtype: str = "bf16", *,
                      out=None, stream=None):
    """Dequantize codes [M, K or K/2] (uint8, CUDA) with their scales (as
    per_token_cast returns them): code value x scale, BF16 or fp32 [M, K]."""
    import torch
    M = codes.shape[0]
    if out is None:
        dt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
        out = torch.empty((M, K), dtype=dt, device=codes.device)
    if stream is None:
        stream = torch.cuda.current_stream(codes.device).cuda_stream
    tk_per_token_dequant(codes.data_ptr(), codes.stride(0), scales.data_ptr(),
                         scales.stride(0), M, K, group, FMT[fmt], SCALE[scale],
                         LAYOUT[layout], out.data_ptr(), out.stride(0),
                         OUT_DTYPE[out_dtype], stream)
    return out


def per_token_cast_back(x, group: int = 128, fmt: str = "e4m3",
                        scale: str = "fp32", *, out=None, stream=None):
    """Quantize then dequantize a bfloat16 [M, K] CUDA tensor in one pass:
    the BF16 values its per-token cast represents."""
    import torch
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bfloat16 tensor with unit column "
                         "stride")
    M, K = x.shape
    if out is None:
        out = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    tk_per_token_cast_back(x.data_ptr(), M, K, x.stride(0), group, FMT[fmt],
                           SCALE[scale], out.data_ptr(), out.stride(0), stream)
    return out


BLOCK = 128   # edge of the per-block cast's square blocks (TK_BLOCK)


def block_scale_shape(M: int, K: int, scale: str = "fp32"):
    """Shape and torch dtype name of the per-block scale tensor."""
    nr, nc = -(-M // BLOCK), -(-K // BLOCK)
    if scale == "ue8m0":
        return (nr, (nc + 3) // 4), "int32"
    return (nr, nc), "float32"


def channel_scale_shape(K: int, scale: str = "fp32"):
    """Shape and torch dtype name of the per-channel scale vector."""
    if scale == "ue8m0":
        return ((K + 3) // 4,), "int32"
    return (K,), "float32"


def _check_x(x):
    import torch
    if (x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1
            or x.device.type != "cuda"):
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor with unit "
                         "column stride")


def _codes(torch, x, fmt, codes):
    if codes is None:
        M, K = x.shape
        codes = _code_buffer(torch, M, K, fmt, x.device)
    return codes


def per_block_cast(x, fmt: str = "e4m3", scale: str = "fp32", *, codes=None,
                   scales=None, stream=None):
    """Per-block cast of a bfloat16 [M, K] CUDA tensor: one scale per
    128 x 128 block.  Returns (codes [M, K or K/2], scales, see
    ``block_scale_shape``); asynchronous on the current stream."""
    import torch
    _check_x(x)
    M, K = x.shape
    codes = _codes(torch, x, fmt, codes)
    if scales is None:
        shape, dt = block_scale_shape(M, K, scale)
        scales = torch.empty(shape, dtype=getattr(torch, dt), device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    tk_per_block_cast(x.data_ptr(), M, K, x.stride(0), FMT[fmt], SCALE[scale],
                      codes.data_ptr(), codes.stride(0), scales.data_ptr(),
                      scales.stride(0), stream)
    return codes, scales


_workspaces = {}


def channel_workspace(K: int, device=None, stream=None):
    """A zero-filled per-channel workspace of at least
    ``tk_per_channel_workspace_bytes(K)`` bytes, kept per (device, stream):
    every completed call leaves it zero-filled, so calls issued on one
    stream can share it (calls on different streams get different ones)."""
    import torch
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    need = max(16, tk_per_channel_workspace_bytes(K))
    key = (dev.index, stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def per_channel_cast(x, fmt: str = "e4m3", scale: str = "fp32", *,
                     codes=None, scales=None, workspace=None, stream=None):
    """Per-channel cast of a bfloat16 [M, K] CUDA tensor: one scale per
    column over all rows.  Returns (codes, scale vector, see
    ``channel_scale_shape``).  ``workspace`` (a zero-filled uint8 CUDA
    tensor of at least ``tk_per_channel_workspace_bytes(K)`` bytes, left
    zero-filled by the call) defaults to ``channel_workspace`` for the
    call's device and stream."""
    import torch
    _check_x(x)
    M, K = x.shape
    codes = _codes(torch, x, fmt, codes)
    if scales is None:
        shape, dt = channel_scale_shape(K, scale)
        scales = torch.empty(shape, dtype=getattr(torch, dt), device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    if workspace is None:
        workspace = channel_workspace(K, x.device, stream)
    tk_per_channel_cast(x.data_ptr(), M, K, x.stride(0), FMT[fmt],
                        SCALE[scale], codes.data_ptr(), codes.stride(0),
                        scales.data_ptr(), workspace.data_ptr(),
                        workspace.numel(), stream)
    return codes, scales


def _dequant_out(torch, codes, K, out_dtype, out):
    if out is None:
        dt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
        out = torch.empty((codes.shape[0], K), dtype=dt, device=codes.device)
    return out


def per_block_dequant(codes, scales, K: int, fmt: str = "e4m3",
                      scale: str = "fp32", out_dtype: str = "bf16", *,
                      out=None, stream=None):
    """Dequantize per-block codes [M, K or K/2] (uint8, CUDA) with the
    scales per_block_cast returns: BF16 or fp32 [M, K]."""
    import torch
    out = _dequant_out(torch, codes, K, out_dtype, out)
    if stream is None:
        stream = torch.cuda.current_stream(codes.device).cuda_stream
    tk_per_block_dequant(codes.data_ptr(), codes.stride(0), scales.data_ptr(),
                         scales.stride(0), codes.shape[0], K, FMT[fmt],
                         SCALE[scale], out.data_ptr(), out.stride(0),
                         OUT_DTYPE[out_dtype], stream)
    return out


def per_channel_dequant(codes, scales, K: int, fmt: str = "e4m3",
                        scale: str = "fp32", out_dtype: str = "bf16", *,
                        out=None, stream=None):
    """Dequantize per-channel codes [M, K or K/2] (uint8, CUDA) with the
    scale vector per_channel_cast returns: BF16 or fp32 [M, K]."""
    import torch
    out = _dequant_out(torch, codes, K, out_dtype, out)
    if stream is None:
        stream = torch.cuda.current_stream(codes.device).cuda_stream
    tk_per_channel_dequant(codes.data_ptr(), codes.stride(0),
                           scales.data_ptr(), codes.shape[0], K, FMT[fmt],
                           SCALE[scale], out.data_ptr(), out.stride(0),
                           OUT_DTYPE[out_dtype], stream)
    return out
