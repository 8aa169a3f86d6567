"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before any CUDA call (CPU only: no kernel runs)."""
import ctypes
import glob
import os
import re

import pytest

import precision_quantization_token_gb300 as tk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3
A = 0x10000          # fake, 16-byte aligned "device" addresses: never touched
B = 0x20000
C = 0x30000


@pytest.fixture(scope="module")
def lib():
    tk.build()
    return tk.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(tk_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "tk_per_token_cast" in names and "tk_swiglu_per_token_cast" in names
    assert "tk_per_block_cast" in names and "tk_per_channel_cast" in names
    raw = ctypes.CDLL(tk.library_path())
    for n in names:
        assert hasattr(raw, n), n


def test_header_is_plain_c(tmp_path):
    """include/*.h is a C ABI: a C99 translation unit (all warnings as
    errors) includes it and takes the address of every declared function."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "abi_check.c"
    src.write_text('#include "tk_cast.h"\n'
                   "void *table[] = {\n" +
                   "".join(f"    (void *)&{n},\n" for n in names) +
                   "};\n")
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror",
                        "-Wno-pedantic", "-fsyntax-only",
                        f"-I{os.path.join(ROOT, 'include')}", str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(lib):
    assert tk.tk_status_string(0) == "TK_OK"
    assert tk.tk_status_string(3) == "TK_ERR_MISALIGNED"
    assert tk.tk_status_string(99) == "TK_ERR_UNKNOWN"
    assert lib.tk_last_cuda_error() == b""


def call(lib, *, x=A, M=4, K=256, ld_x=256, group=128, fmt=0, mode=0,
         layout=0, codes=B, ld_codes=256, scales=C, ld_scales=2, swiglu=False):
    fn = lib.tk_swiglu_per_token_cast if swiglu else lib.tk_per_token_cast
    return fn(x, M, K, ld_x, group, fmt, mode, layout, codes, ld_codes, scales,
              ld_scales, None)


CASES = [
    ("bad group", dict(group=48), INVALID),
    ("group 8", dict(group=8), INVALID),
    ("K not multiple of group", dict(K=200, ld_x=256), INVALID),
    ("K zero", dict(K=0), INVALID),
    ("negative M", dict(M=-1), INVALID),
    ("bad fmt", dict(fmt=2), INVALID),
    ("bad mode", dict(mode=3), INVALID),
    ("bad layout", dict(layout=2), INVALID),
    ("ld_x < K", dict(ld_x=128), INVALID),
    ("ld_codes < K", dict(ld_codes=128), INVALID),
    ("e2m1 ld_codes < K/2", dict(fmt=1, ld_codes=112), INVALID),
    ("row scales too narrow", dict(ld_scales=1), INVALID),
    ("packed scales too narrow", dict(mode=2, K=1280, ld_x=1280,
                                      ld_codes=1280, ld_scales=2), INVALID),
    ("transposed ld < M", dict(layout=1, M=8, ld_scales=4), INVALID),
    ("null x", dict(x=None), INVALID),
    ("null codes", dict(codes=None), INVALID),
    ("null scales", dict(scales=None), INVALID),
    ("x misaligned", dict(x=A + 8), MISALIGNED),
    ("ld_x not 16 bytes", dict(K=128, ld_x=132), MISALIGNED),
    ("codes misaligned", dict(codes=B + 4), MISALIGNED),
    ("ld_codes not 16", dict(ld_codes=264), MISALIGNED),
    ("scales misaligned", dict(scales=C + 2), MISALIGNED),
    ("transposed ld not multiple of 4", dict(layout=1, M=5, ld_scales=5),
     MISALIGNED),
    ("M too large", dict(M=(1 << 30) + 1), UNSUPPORTED),
    ("K too large", dict(K=(1 << 28) + 128, ld_x=(1 << 28) + 128,
                         ld_codes=(1 << 28) + 128, ld_scales=1 << 22),
     UNSUPPORTED),
    ("swiglu ld_x < 2N", dict(swiglu=True, ld_x=384), INVALID),
]


@pytest.mark.parametrize("name,kw,want", CASES, ids=[c[0] for c in CASES])
def test_validation(lib, name, kw, want):
    assert call(lib, **kw) == want


def call_dq(lib, *, codes=A, ld_codes=256, scales=C, ld_scales=2, M=4, K=256,
            group=128, fmt=0, mode=0, layout=0, y=B, ld_y=256, out=0):
    return lib.tk_per_token_dequant(codes, ld_codes, scales, ld_scales, M, K,
                                    group, fmt, mode, layout, y, ld_y, out,
                                    None)


DQ_CASES = [
    ("bad out dtype", dict(out=2), INVALID),
    ("bad group", dict(group=8), INVALID),
    ("ld_codes < K", dict(ld_codes=128), INVALID),
    ("ld_y < K", dict(ld_y=128), INVALID),
    ("scales too narrow", dict(ld_scales=1), INVALID),
    ("null y", dict(y=None), INVALID),
    ("null codes", dict(codes=None), INVALID),
    ("codes misaligned", dict(codes=A + 8), MISALIGNED),
    ("y misaligned", dict(y=B + 4), MISALIGNED),
    ("bf16 ld_y not 16 bytes", dict(K=128, ld_y=132, ld_scales=1), MISALIGNED),
    ("fp32 ld_y not 16 bytes", dict(K=128, ld_y=130, ld_scales=1, out=1),
     MISALIGNED),
    ("transposed ld not multiple of 4", dict(layout=1, M=5, ld_scales=5),
     MISALIGNED),
    ("M too large", dict(M=(1 << 30) + 1), UNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,want", DQ_CASES, ids=[c[0] for c in DQ_CASES])
def test_dequant_validation(lib, name, kw, want):
    assert call_dq(lib, **kw) == want


def call_cb(lib, *, x=A, M=4, K=256, ld_x=256, group=128, fmt=0, mode=0,
            y=B, ld_y=256):
    return lib.tk_per_token_cast_back(x, M, K, ld_x, group, fmt, mode, y,
                                      ld_y, None)


CB_CASES = [
    ("bad mode", dict(mode=5), INVALID),
    ("K not multiple of group", dict(K=200), INVALID),
    ("ld_y < K", dict(ld_y=128), INVALID),
    ("null x", dict(x=None), INVALID),
    ("y misaligned", dict(y=B + 2), MISALIGNED),
    ("ld_y not 16 bytes", dict(K=128, ld_x=128, ld_y=132), MISALIGNED),
]


@pytest.mark.parametrize("name,kw,want", CB_CASES, ids=[c[0] for c in CB_CASES])
def test_cast_back_validation(lib, name, kw, want):
    assert call_cb(lib, **kw) == want


def call_pb(lib, *, x=A, M=4, K=256, ld_x=256, fmt=0, mode=0, codes=B,
            ld_codes=256, scales=C, ld_scales=2):
    return lib.tk_per_block_cast(x, M, K, ld_x, fmt, mode, codes, ld_codes,
                                 scales, ld_scales, None)


PB_CASES = [
    ("bad fmt", dict(fmt=2), INVALID),
    ("bad mode", dict(mode=3), INVALID),
    ("K not multiple of 16", dict(K=200, ld_x=256), INVALID),
    ("K zero", dict(K=0), INVALID),
    ("negative M", dict(M=-1), INVALID),
    ("ld_x < K", dict(ld_x=128), INVALID),
    ("ld_codes < K", dict(ld_codes=128), INVALID),
    ("e2m1 ld_codes < K/2", dict(fmt=1, ld_codes=112), INVALID),
    ("scale row too narrow", dict(ld_scales=1), INVALID),
    ("ragged K needs another word", dict(K=272, ld_x=272, ld_codes=272,
                                         ld_scales=2), INVALID),
    ("packed scale row too narrow", dict(mode=2, K=1280, ld_x=1280,
                                         ld_codes=1280, ld_scales=2), INVALID),
    ("null x", dict(x=None), INVALID),
    ("null codes", dict(codes=None), INVALID),
    ("null scales", dict(scales=None), INVALID),
    ("x misaligned", dict(x=A + 8), MISALIGNED),
    ("ld_x not 16 bytes", dict(K=128, ld_x=132, ld_scales=1), MISALIGNED),
    ("codes misaligned", dict(codes=B + 4), MISALIGNED),
    ("ld_codes not 16", dict(ld_codes=264), MISALIGNED),
    ("scales misaligned", dict(scales=C + 2), MISALIGNED),
    ("M too large", dict(M=(1 << 30) + 1), UNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,want", PB_CASES, ids=[c[0] for c in PB_CASES])
def test_per_block_validation(lib, name, kw, want):
    assert call_pb(lib, **kw) == want


WS = 0x40000


def call_pc(lib, *, x=A, M=4, K=256, ld_x=256, fmt=0, mode=0, codes=B,
            ld_codes=256, scales=C, ws=WS, ws_bytes=4 * 256 + 16):
    return lib.tk_per_channel_cast(x, M, K, ld_x, fmt, mode, codes, ld_codes,
                                   scales, ws, ws_bytes, None)


PC_CASES = [
    ("bad fmt", dict(fmt=2), INVALID),
    ("bad mode", dict(mode=7), INVALID),
    ("K not multiple of 16", dict(K=120, ld_x=128), INVALID),
    ("ld_x < K", dict(ld_x=128), INVALID),
    ("ld_codes < K", dict(ld_codes=128), INVALID),
    ("workspace too small", dict(ws_bytes=4 * 256 + 15), INVALID),
    ("workspace for padded K", dict(K=272, ld_x=272, ld_codes=272,
                                    ws_bytes=4 * 384 + 15), INVALID),
    ("null workspace", dict(ws=None), INVALID),
    ("null x", dict(x=None), INVALID),
    ("null scales", dict(scales=None), INVALID),
    ("workspace misaligned", dict(ws=WS + 8), MISALIGNED),
    ("x misaligned", dict(x=A + 8), MISALIGNED),
    ("scales misaligned", dict(scales=C + 1), MISALIGNED),
    ("K too large", dict(K=(1 << 28) + 16, ld_x=(1 << 28) + 16,
                         ld_codes=(1 << 28) + 16, ws_bytes=1 << 40), UNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,want", PC_CASES, ids=[c[0] for c in PC_CASES])
def test_per_channel_validation(lib, name, kw, want):
    assert call_pc(lib, **kw) == want


def call_na(lib, *, x=A, M=4, K=256, ld_x=256, fmt=0, mode=0, codes=B,
            ld_codes=256, scales=C):
    return lib.tk_per_channel_cast_noalloc(x, M, K, ld_x, fmt, mode, codes,
                                           ld_codes, scales, None)


NA_CASES = [
    ("bad fmt", dict(fmt=2), INVALID),
    ("bad mode", dict(mode=3), INVALID),
    ("K not multiple of 16", dict(K=200, ld_x=256), INVALID),
    ("ld_codes < K", dict(ld_codes=128), INVALID),
    ("null x", dict(x=None), INVALID),
    ("x misaligned", dict(x=A + 8), MISALIGNED),
    ("scales misaligned", dict(scales=C + 2), MISALIGNED),
    ("beyond the static workspace", dict(K=65536 + 16, ld_x=65536 + 16,
                                         ld_codes=65536 + 16), UNSUPPORTED),
    ("beyond it even with M = 0", dict(M=0, K=65536 + 16, ld_x=65536 + 16,
                                       ld_codes=65536 + 16), UNSUPPORTED),
    ("empty batch", dict(M=0, x=None, codes=None, scales=None), OK),
]


@pytest.mark.parametrize("name,kw,want", NA_CASES, ids=[c[0] for c in NA_CASES])
def test_per_channel_noalloc_validation(lib, name, kw, want):
    assert call_na(lib, **kw) == want


def call_rms(lib, *, x=A, w=WS, M=4, K=256, ld_x=256, eps=1e-6, group=128,
             fmt=0, mode=0, layout=0, codes=B, ld_codes=256, scales=C,
             ld_scales=2):
    return lib.tk_rmsnorm_per_token_cast(x, w, M, K, ld_x, eps, group, fmt,
                                         mode, layout, codes, ld_codes,
                                         scales, ld_scales, None)


RMS_CASES = [
    ("bad group", dict(group=48), INVALID),
    ("negative eps", dict(eps=-1e-6), INVALID),
    ("nan eps", dict(eps=float("nan")), INVALID),
    ("inf eps", dict(eps=float("inf")), INVALID),
    ("ld_x < K", dict(ld_x=128), INVALID),
    ("scales too narrow", dict(ld_scales=1), INVALID),
    ("null gain", dict(w=None), INVALID),
    ("gain misaligned", dict(w=WS + 8), MISALIGNED),
    ("x misaligned", dict(x=A + 8), MISALIGNED),
    ("row longer than a stage", dict(K=8192 + 128, ld_x=8320, ld_codes=8320,
                                     ld_scales=65), UNSUPPORTED),
    ("empty batch", dict(M=0, x=None, w=None, codes=None, scales=None), OK),
    ("zero eps allowed", dict(M=0, eps=0.0), OK),
]


@pytest.mark.parametrize("name,kw,want", RMS_CASES, ids=[c[0] for c in RMS_CASES])
def test_rmsnorm_validation(lib, name, kw, want):
    assert call_rms(lib, **kw) == want


def call_bd(lib, *, codes=A, ld_codes=256, scales=C, ld_scales=2, M=4,
            K=256, fmt=0, mode=0, y=B, ld_y=256, out=0):
    return lib.tk_per_block_dequant(codes, ld_codes, scales, ld_scales, M, K,
                                    fmt, mode, y, ld_y, out, None)


def call_cd(lib, *, codes=A, ld_codes=256, scales=C, M=4, K=256, fmt=0,
            mode=0, y=B, ld_y=256, out=0):
    return lib.tk_per_channel_dequant(codes, ld_codes, scales, M, K, fmt, mode,
                                      y, ld_y, out, None)


TILE_DQ_CASES = [
    ("block bad out dtype", call_bd, dict(out=2), INVALID),
    ("block K not multiple of 16", call_bd, dict(K=200), INVALID),
    ("block scale row too narrow", call_bd, dict(ld_scales=1), INVALID),
    ("block ld_y < K", call_bd, dict(ld_y=128), INVALID),
    ("block codes misaligned", call_bd, dict(codes=A + 8), MISALIGNED),
    ("block scales misaligned", call_bd, dict(scales=C + 2), MISALIGNED),
    ("block fp32 ld_y not 16 bytes", call_bd, dict(K=128, ld_y=130,
                                                   ld_scales=1, out=1), MISALIGNED),
    ("block empty batch", call_bd, dict(M=0, codes=None, scales=None, y=None), OK),
    ("channel bad fmt", call_cd, dict(fmt=3), INVALID),
    ("channel ld_codes < K", call_cd, dict(ld_codes=128), INVALID),
    ("channel null scales", call_cd, dict(scales=None), INVALID),
    ("channel scales not 16-byte aligned", call_cd, dict(scales=C + 4), MISALIGNED),
    ("channel y misaligned", call_cd, dict(y=B + 2), MISALIGNED),
    ("channel M too large", call_cd, dict(M=(1 << 30) + 1), UNSUPPORTED),
    ("channel empty batch", call_cd, dict(M=0, codes=None, scales=None, y=None), OK),
]


@pytest.mark.parametrize("name,fn,kw,want", TILE_DQ_CASES,
                         ids=[c[0] for c in TILE_DQ_CASES])
def test_tile_dequant_validation(lib, name, fn, kw, want):
    assert fn(lib, **kw) == want


def test_per_channel_workspace_size(lib):
    # maxima for K rounded up to 128 channels + one counter per 128 (16-B units)
    assert tk.tk_per_channel_workspace_bytes(256) == 4 * 256 + 16
    assert tk.tk_per_channel_workspace_bytes(16) == 4 * 128 + 16
    assert tk.tk_per_channel_workspace_bytes(7168) == 4 * 7168 + 224
    assert tk.tk_per_channel_workspace_bytes(8 * 128 + 16) == 4 * 9 * 128 + 48
    assert tk.tk_per_channel_workspace_bytes(0) == 0
    assert tk.tk_per_channel_workspace_bytes(-5) == 0


def call_host(lib, *, x=A, M=4, K=256, ld_x=256, group=128, fmt=0, mode=0,
              layout=0, codes=B, ld_codes=256, scales=C, ld_scales=2,
              scratch=0x40000, scratch_bytes=1 << 20, chunk_rows=0,
              n_streams=2, swiglu=False, no_array=False):
    fn = (lib.tk_swiglu_per_token_cast_host if swiglu
          else lib.tk_per_token_cast_host)
    arr = None if no_array else (ctypes.c_void_p * max(n_streams, 1))()
    return fn(x, M, K, ld_x, group, fmt, mode, layout, codes, ld_codes, scales,
              ld_scales, scratch, scratch_bytes, chunk_rows, arr, n_streams)


HOST_CASES = [
    ("bad group", dict(group=48), INVALID),
    ("bad layout", dict(layout=2), INVALID),
    ("ld_x < K", dict(ld_x=128), INVALID),
    ("swiglu ld_x < 2N", dict(swiglu=True, ld_x=256), INVALID),
    ("ld_codes < K", dict(ld_codes=255), INVALID),
    ("ld_scales < G", dict(ld_scales=1), INVALID),
    ("transposed ld_scales < M", dict(layout=1, ld_scales=3), INVALID),
    ("negative chunk_rows", dict(chunk_rows=-1), INVALID),
    ("no streams", dict(n_streams=0), INVALID),
    ("65 streams", dict(n_streams=65), INVALID),
    ("null stream array", dict(no_array=True), INVALID),
    ("null x", dict(x=None), INVALID),
    ("null scales", dict(scales=None), INVALID),
    ("null scratch", dict(scratch=None), INVALID),
    ("scratch too small", dict(scratch_bytes=1024), INVALID),
    ("scratch misaligned", dict(scratch=0x40008), MISALIGNED),
    ("empty batch", dict(M=0, x=None, codes=None, scales=None, scratch=None,
                         scratch_bytes=0), OK),
    ("too many rows", dict(M=(1 << 30) + 1), UNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,want", HOST_CASES, ids=[c[0] for c in HOST_CASES])
def test_host_entry_validation(lib, name, kw, want):
    """Host buffers take no alignment rule: only the device scratch must be
    aligned; every check fails before any copy or launch."""
    assert call_host(lib, **kw) == want


def test_host_scratch_size(lib):
    """Input rows padded to 16 B, code rows to 16 B, row-major scale rows
    unpadded (transposed: tokens padded to 4), each region rounded up to
    256 B."""
    def r256(v):
        return (v + 255) // 256 * 256
    # 4096 x 7168 E4M3 g128 UE8M0 row-major: 14 words per row
    assert tk.tk_host_scratch_bytes(4096, 7168, 128, 0, 2, 0, 0) == (
        4096 * 7168 * 2 + 4096 * 7168 + r256(4096 * 14 * 4))
    # SwiGLU 3 x [272 | 272] E2M1 g16 fp32 transposed: 17 scale rows x 4
    assert tk.tk_host_scratch_bytes(3, 272, 16, 1, 0, 1, 1) == (
        r256(3 * 544 * 2) + r256(3 * 144) + r256(17 * 4 * 4))
    # 5 x 272 E2M1 g16 fp32 row-major: 17 words per row
    assert tk.tk_host_scratch_bytes(5, 272, 16, 1, 0, 0, 0) == (
        r256(5 * 272 * 2) + r256(5 * 144) + r256(5 * 17 * 4))
    assert tk.tk_host_scratch_bytes(4, 200, 128, 0, 0, 0, 0) == 0   # K % group
    assert tk.tk_host_scratch_bytes(4, 256, 128, 0, 0, 0, 1) == (
        r256(4 * 512 * 2) + r256(4 * 256) + r256(4 * 2 * 4))


def test_empty_batch_is_a_noop(lib):
    assert call_pb(lib, M=0, x=None, codes=None, scales=None) == OK
    assert call_pc(lib, M=0, x=None, codes=None, scales=None, ws=None) == OK
    assert call_dq(lib, M=0, codes=None, scales=None, y=None) == OK
    assert call_cb(lib, M=0, x=None, y=None) == OK
    assert call(lib, M=0, x=None, codes=None, scales=None) == OK
    assert call(lib, M=0, x=None, codes=None, scales=None, swiglu=True,
                ld_x=512) == OK


def test_fault_query_rejects_null(lib):
    assert lib.tk_get_device_fault(None, 0) == INVALID


def test_python_wrapper_raises(lib):
    with pytest.raises(tk.TkError) as e:
        tk.tk_per_token_cast(A, 4, 256, 256, 48, 0, 0, 0, B, 256, C, 2, 0)
    assert e.value.status == INVALID


def test_product_package_does_not_touch_the_oracle():
    """The product package imports nothing from oracle/ (and vice versa)."""
    pkg = os.path.join(ROOT, "precision_quantization_token_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            src = open(path).read()
            assert not re.search(r"^\s*(import|from)\s+oracle", src, re.M), path
            assert "tk_oracle" not in src, path
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.*")):
        if path.endswith((".py", ".c")):
            src = open(path).read()
            assert "import precision_quantization_token_gb300" not in src
            assert "from precision_quantization_token_gb300" not in src
            assert "tk_cast.h" not in src
