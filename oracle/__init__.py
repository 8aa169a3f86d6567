"""Plain CPU oracle of the per-token group-wise cast (test infrastructure).

This package is TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it.  The product library
(``precision_quantization_token_gb300``) never imports, loads or calls it, and
it imports nothing from the product library: the two share no code.

The arithmetic lives in ``tk_oracle.c`` (plain C11, scalar, compiled with
``-O2 -ffp-contract=off`` and no fast-math so that every ``a / b`` is one IEEE
fp32 division).  This module only builds it with gcc, loads it with ctypes and
splits rows across host threads (ctypes releases the GIL during each call, and
the C code writes disjoint rows, so the split does not change any result).

Sources followed (see tk_oracle.c for the per-step notes):
  * TileKernels README (tile-kernels 2.0.0 on PyPI), "Features": per-token
    FP8/FP4 casting and fused SwiGLU+quantization.
  * aiwiki "TileKernels", "Quantization": groups of 16/32/64/128 channels,
    power-of-two scale rounding, packed UE8M0 scales, per-token scales in
    DeepGEMM's (transposed, M-padded) layout.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tk_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libtk_oracle.so")

FMT_E4M3, FMT_E2M1 = 0, 1
SCALE_FP32, SCALE_FP32_POW2, SCALE_UE8M0 = 0, 1, 2
LAYOUT_ROW_MAJOR, LAYOUT_TRANSPOSED = 0, 1

_lib = None
_lock = threading.Lock()
_pool = None
_pool_size = 0


def build(force: bool = False) -> str:
    """Compile tk_oracle.c into a shared library with gcc; returns its path."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    i64, p, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    sig = [p, i64, i64, i64, i64, i, i, i, i, p, i64, p, i64]
    lib.oracle_per_token_cast.argtypes = sig
    lib.oracle_per_token_cast.restype = i
    lib.oracle_swiglu_per_token_cast.argtypes = sig
    lib.oracle_swiglu_per_token_cast.restype = i
    lib.oracle_swiglu_value.argtypes = [ctypes.c_float, ctypes.c_float]
    lib.oracle_swiglu_value.restype = ctypes.c_float
    lib.oracle_encode.argtypes = [p, i64, i, p]
    lib.oracle_encode.restype = None
    lib.oracle_scale.argtypes = [p, i64, i, i, p, p]
    lib.oracle_scale.restype = None
    lib.oracle_swiglu_values.argtypes = [p, i64, i64, i64, i64, p, i64]
    lib.oracle_swiglu_values.restype = None
    lib.oracle_per_token_dequant.argtypes = [p, i64, p, i64, i64, i64, i64, i,
                                             i, i, i, i, p, i64]
    lib.oracle_per_token_dequant.restype = i
    lib.oracle_per_token_cast_back.argtypes = [p, i64, i64, i64, i64, i, i, i,
                                               p, i64]
    lib.oracle_per_token_cast_back.restype = i
    lib.oracle_rmsnorm_values.argtypes = [p, p, i64, i64, i64, i64,
                                          ctypes.c_float, p, i64]
    lib.oracle_rmsnorm_values.restype = None
    lib.oracle_rmsnorm_per_token_cast.argtypes = [p, p, i64, i64, i64, i64,
                                                  ctypes.c_float, i, i, i, i,
                                                  p, i64, p, i64]
    lib.oracle_rmsnorm_per_token_cast.restype = i
    lib.oracle_per_block_dequant.argtypes = [p, i64, p, i64, i64, i64, i64,
                                             i, i, i, i, p, i64]
    lib.oracle_per_block_dequant.restype = i
    lib.oracle_per_channel_dequant.argtypes = [p, i64, p, i64, i64, i64, i,
                                               i, i, p, i64]
    lib.oracle_per_channel_dequant.restype = i
    lib.oracle_per_block_cast.argtypes = [p, i64, i64, i64, i, i64, i64, i, i,
                                          p, i64, p, i64]
    lib.oracle_per_block_cast.restype = i
    lib.oracle_per_channel_cast.argtypes = [p, i64, i64, i64, i64, i64, i, i,
                                            p, i64, p]
    lib.oracle_per_channel_cast.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


def compile_variant(src_text: str, out_path: str):
    """Compile an edited copy of the oracle source (used by the tests that
    plant mistakes in the oracle to show that its pins catch them)."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off",
                    "-fno-fast-math", "-fPIC", "-shared", "-w", "-o", out_path,
                    c_path, "-lm"], check=True)
    return _configure(ctypes.CDLL(out_path))


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _executor(threads: int) -> ThreadPoolExecutor:
    """A process-wide thread pool, reused across calls (grown on demand)."""
    global _pool, _pool_size
    with _lock:
        if _pool is None or _pool_size < threads:
            if _pool is not None:
                _pool.shutdown(wait=False)
            _pool = ThreadPoolExecutor(threads)
            _pool_size = threads
        return _pool


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def scale_shape(M: int, K: int, group: int, mode: int, layout: int,
                m_pad_to: int = 4):
    """(rows, cols, dtype) of the scale tensor for an [M, K] cast.

    Row-major: [M, G] fp32 or [M, ceil(G/4)] int32 (packed UE8M0).
    Transposed ("DeepGEMM's layout"): [G, M_pad] fp32 or [ceil(G/4), M_pad]
    int32, with M_pad = ceil(M / m_pad_to) * m_pad_to.
    """
    G = K // group
    cols = (G + 3) // 4 if mode == SCALE_UE8M0 else G
    dtype = np.int32 if mode == SCALE_UE8M0 else np.float32
    if layout == LAYOUT_ROW_MAJOR:
        return M, cols, dtype
    m_pad = (M + m_pad_to - 1) // m_pad_to * m_pad_to
    return cols, m_pad, dtype


def _run(fn, x, n_rows, K_or_N, ld_x, group, fmt, mode, layout, codes,
         scales, threads):
    ld_codes = codes.strides[0]
    ld_scales = scales.strides[0] // scales.itemsize
    threads = max(1, min(threads or 1, n_rows))
    bounds = np.linspace(0, n_rows, threads + 1).astype(np.int64)

    def work(t):
        return fn(_ptr(x), int(bounds[t]), int(bounds[t + 1]), K_or_N, ld_x,
                  group, fmt, mode, layout, _ptr(codes), ld_codes,
                  _ptr(scales), ld_scales)

    if threads == 1:
        rcs = [work(0)]
    else:
        rcs = list(_executor(threads).map(work, range(threads)))
    for rc in rcs:
        if rc != 0:
            raise ValueError(f"oracle returned status {rc}")


def per_token_cast(x_bits: np.ndarray, K: int, group: int, fmt: int, mode: int,
                   layout: int, *, codes: np.ndarray | None = None,
                   scales: np.ndarray | None = None, threads: int = 1):
    """Oracle cast of a BF16 matrix given as uint16 bit patterns [M, ld_x].

    Returns (codes uint8 [M, K or K/2], scales) with the shapes of
    ``scale_shape``.  Pre-filled ``codes``/``scales`` may be passed (their
    untouched entries then keep their contents).
    """
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, ld_x = x_bits.shape
    lib = _load()
    row_bytes = K if fmt == FMT_E4M3 else K // 2
    if codes is None:
        codes = np.zeros((M, row_bytes), np.uint8)
    if scales is None:
        r, c, dt = scale_shape(M, K, group, mode, layout)
        scales = np.zeros((r, c), dt)
    _run(lib.oracle_per_token_cast, x_bits, M, K, ld_x, group, fmt, mode,
         layout, codes, scales, threads)
    return codes, scales


def swiglu_per_token_cast(x_bits: np.ndarray, N: int, group: int, fmt: int,
                          mode: int, layout: int, *, codes=None, scales=None,
                          threads: int = 1):
    """Oracle fused SwiGLU + cast; x_bits is [M, ld_x >= 2N] = [gate | up]."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, ld_x = x_bits.shape
    lib = _load()
    row_bytes = N if fmt == FMT_E4M3 else N // 2
    if codes is None:
        codes = np.zeros((M, row_bytes), np.uint8)
    if scales is None:
        r, c, dt = scale_shape(M, N, group, mode, layout)
        scales = np.zeros((r, c), dt)
    _run(lib.oracle_swiglu_per_token_cast, x_bits, M, N, ld_x, group, fmt,
         mode, layout, codes, scales, threads)
    return codes, scales


def swiglu_values(x_bits: np.ndarray, N: int, threads: int = 1) -> np.ndarray:
    """The fp32 SwiGLU product [M, N] of x_bits = [gate | up] (no cast)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, ld_x = x_bits.shape
    y = np.empty((M, N), np.float32)
    lib = _load()
    threads = max(1, min(threads or 1, M))
    bounds = np.linspace(0, M, threads + 1).astype(np.int64)

    def work(t):
        lib.oracle_swiglu_values(_ptr(x_bits), int(bounds[t]),
                                 int(bounds[t + 1]), N, ld_x, _ptr(y), N)

    if threads == 1:
        work(0)
    else:
        list(_executor(threads).map(work, range(threads)))
    return y


def _split(n_rows, threads, work):
    threads = max(1, min(threads or 1, n_rows)) if n_rows else 1
    bounds = np.linspace(0, n_rows, threads + 1).astype(np.int64)
    jobs = [(int(bounds[t]), int(bounds[t + 1])) for t in range(threads)]
    if threads == 1:
        rcs = [work(*jobs[0])]
    else:
        rcs = list(_executor(threads).map(lambda j: work(*j), jobs))
    for rc in rcs:
        if rc != 0:
            raise ValueError(f"oracle returned status {rc}")


def per_token_dequant(codes: np.ndarray, scales: np.ndarray, K: int,
                      group: int, fmt: int, mode: int, layout: int, *,
                      out_fp32: bool = False, threads: int = 1):
    """Oracle dequantization: code value x scale (one fp32 multiply), as
    fp32 or rounded to BF16 bits.  codes/scales as the cast writes them."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales)
    M = codes.shape[0]
    y = np.zeros((M, K), np.float32 if out_fp32 else np.uint16)
    lib = _load()
    ld_s = scales.strides[0] // scales.itemsize

    def work(a, b):
        return lib.oracle_per_token_dequant(
            _ptr(codes), codes.strides[0], _ptr(scales), ld_s, a, b, K,
            group, fmt, mode, layout, int(out_fp32), _ptr(y), K)

    _split(M, threads, work)
    return y


def per_token_cast_back(x_bits: np.ndarray, K: int, group: int, fmt: int,
                        mode: int, *, threads: int = 1) -> np.ndarray:
    """Oracle cast-and-cast-back: BF16 bits in, BF16 bits out."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, ld_x = x_bits.shape
    y = np.zeros((M, K), np.uint16)
    lib = _load()

    def work(a, b):
        return lib.oracle_per_token_cast_back(_ptr(x_bits), a, b, K, ld_x,
                                              group, fmt, mode, _ptr(y), K)

    _split(M, threads, work)
    return y


def rmsnorm_values(x_bits: np.ndarray, w_bits: np.ndarray, K: int,
                   eps: float, threads: int = 1) -> np.ndarray:
    """RMSNorm outputs y (fp32 [M, K]) of BF16 rows x with gain w."""
    lib = _load()
    M = x_bits.shape[0]
    ld_x = x_bits.strides[0] // 2
    w_bits = np.ascontiguousarray(w_bits, np.uint16)
    y = np.empty((M, K), np.float32)

    def work(a, b):
        lib.oracle_rmsnorm_values(_ptr(x_bits), _ptr(w_bits), a, b, K, ld_x,
                                  eps, _ptr(y), K)
        return 0

    _split(M, threads, work)
    return y


def rmsnorm_per_token_cast(x_bits: np.ndarray, w_bits: np.ndarray, K: int,
                           eps: float, group: int, fmt: int, mode: int,
                           layout: int, *, codes: np.ndarray | None = None,
                           scales: np.ndarray | None = None,
                           threads: int = 1):
    """Oracle RMSNorm (gain w, eps) fused with the per-token cast of its
    fp32 output.  Shapes as for ``per_token_cast``."""
    lib = _load()
    M = x_bits.shape[0]
    ld_x = x_bits.strides[0] // 2
    w_bits = np.ascontiguousarray(w_bits, np.uint16)
    if codes is None:
        codes = np.zeros((M, K if fmt == FMT_E4M3 else K // 2), np.uint8)
    if scales is None:
        r, c, dt = scale_shape(M, K, group, mode, layout)
        scales = np.zeros((r, c), dt)
    ld_codes = codes.strides[0]
    ld_scales = scales.strides[0] // scales.itemsize

    def work(a, b):
        return lib.oracle_rmsnorm_per_token_cast(
            _ptr(x_bits), _ptr(w_bits), a, b, K, ld_x, eps, group, fmt, mode,
            layout, _ptr(codes), ld_codes, _ptr(scales), ld_scales)

    _split(M, threads, work)
    return codes, scales


def block_scale_shape(M: int, K: int, block: int, mode: int):
    """(rows, cols, dtype) of the per-block scale tensor: one row per block
    row, one fp32 word per block column or ceil(blocks / 4) packed UE8M0
    words."""
    nr = (M + block - 1) // block
    nc = (K + block - 1) // block
    if mode == SCALE_UE8M0:
        return nr, (nc + 3) // 4, np.int32
    return nr, nc, np.float32


def channel_scale_shape(K: int, mode: int):
    """(length, dtype) of the per-channel scale vector."""
    if mode == SCALE_UE8M0:
        return (K + 3) // 4, np.int32
    return K, np.float32


def _codes_for(M, K, fmt, codes):
    if codes is None:
        codes = np.zeros((M, K if fmt == FMT_E4M3 else K // 2), np.uint8)
    return codes


def _check(rcs):
    for rc in rcs:
        if rc != 0:
            raise ValueError(f"oracle returned status {rc}")


def per_block_cast(x_bits: np.ndarray, K: int, block: int, fmt: int,
                   mode: int, *, codes: np.ndarray | None = None,
                   scales: np.ndarray | None = None, threads: int = 1):
    """Oracle per-block cast (square blocks of ``block`` rows x channels) of
    a BF16 matrix given as uint16 bit patterns [M, ld_x].  Returns (codes,
    scales) with scales shaped by ``block_scale_shape``; block rows are
    split across host threads."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits) if x_bits.strides[1] != 2 else x_bits
    M = x_bits.shape[0]
    ld_x = x_bits.strides[0] // 2
    codes = _codes_for(M, K, fmt, codes)
    if scales is None:
        r, c, dt = block_scale_shape(M, K, block, mode)
        scales = np.zeros((r, c), dt)
    n_rb = (M + block - 1) // block
    threads = max(1, min(threads or 1, n_rb))
    bounds = np.linspace(0, n_rb, threads + 1).astype(np.int64)
    ld_s = scales.strides[0] // 4

    def work(t):
        return lib.oracle_per_block_cast(
            _ptr(x_bits), M, K, ld_x, block, int(bounds[t]),
            int(bounds[t + 1]), fmt, mode, _ptr(codes), codes.strides[0],
            _ptr(scales), ld_s)

    _check([work(0)] if threads == 1 else
           list(_executor(threads).map(work, range(threads))))
    return codes, scales


def per_channel_cast(x_bits: np.ndarray, K: int, fmt: int, mode: int, *,
                     codes: np.ndarray | None = None,
                     scales: np.ndarray | None = None, threads: int = 1):
    """Oracle per-channel cast (one scale per channel over all rows) of a
    BF16 matrix given as uint16 bit patterns [M, ld_x].  Returns (codes,
    scale vector shaped by ``channel_scale_shape``); channels are split
    across host threads in multiples of 8."""
    lib = _load()
    M = x_bits.shape[0]
    ld_x = x_bits.strides[0] // 2
    codes = _codes_for(M, K, fmt, codes)
    if scales is None:
        n, dt = channel_scale_shape(K, mode)
        scales = np.zeros(n, dt)
    n8 = (K + 7) // 8
    threads = max(1, min(threads or 1, n8))
    bounds = [min(K, 8 * b) for b in
              np.linspace(0, n8, threads + 1).astype(np.int64)]

    def work(t):
        return lib.oracle_per_channel_cast(
            _ptr(x_bits), M, K, ld_x, int(bounds[t]), int(bounds[t + 1]),
            fmt, mode, _ptr(codes), codes.strides[0], _ptr(scales))

    _check([work(0)] if threads == 1 else
           list(_executor(threads).map(work, range(threads))))
    return codes, scales


def _dequant_out(M, K, out_fp32):
    return np.zeros((M, K), np.float32 if out_fp32 else np.uint16)


def per_block_dequant(codes: np.ndarray, scales: np.ndarray, K: int,
                      block: int, fmt: int, mode: int, *,
                      out_fp32: bool = False, threads: int = 1):
    """Oracle per-block dequantization (codes and scales as per_block_cast
    returns them): fp32, or BF16 bits."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales)
    M = codes.shape[0]
    y = _dequant_out(M, K, out_fp32)
    ld_s = scales.strides[0] // 4

    def work(a, b):
        return lib.oracle_per_block_dequant(
            _ptr(codes), codes.strides[0], _ptr(scales), ld_s, a, b, K, block,
            fmt, mode, int(out_fp32), _ptr(y), K)

    _split(M, threads, work)
    return y


def per_channel_dequant(codes: np.ndarray, scales: np.ndarray, K: int,
                        fmt: int, mode: int, *, out_fp32: bool = False,
                        threads: int = 1):
    """Oracle per-channel dequantization (codes and the scale vector as
    per_channel_cast returns them): fp32, or BF16 bits."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales)
    M = codes.shape[0]
    y = _dequant_out(M, K, out_fp32)

    def work(a, b):
        return lib.oracle_per_channel_dequant(
            _ptr(codes), codes.strides[0], _ptr(scales), a, b, K, fmt, mode,
            int(out_fp32), _ptr(y), K)

    _split(M, threads, work)
    return y


def swiglu_value(gate: float, up: float) -> float:
    return float(_load().oracle_swiglu_value(gate, up))


def encode(q: np.ndarray, fmt: int) -> np.ndarray:
    """Saturating round-to-nearest-even encode of fp32 values."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    out = np.empty(q.shape, np.uint8)
    _load().oracle_encode(_ptr(q), q.size, fmt, _ptr(out))
    return out


def scale(amax: np.ndarray, fmt: int, mode: int):
    """Scale step alone: returns (fp32 scale, UE8M0 byte or -1)."""
    amax = np.ascontiguousarray(amax, dtype=np.float32)
    s = np.empty(amax.shape, np.float32)
    e = np.empty(amax.shape, np.int32)
    _load().oracle_scale(_ptr(amax), amax.size, fmt, mode, _ptr(s), _ptr(e))
    return s, e


def host_threads() -> int:
    return os.cpu_count() or 1
