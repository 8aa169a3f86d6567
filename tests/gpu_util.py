"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
guarded, strided buffers, run the oracle on identical host buffers, and
compare.  Test infrastructure: imports both sides, shares no arithmetic."""
from __future__ import annotations

import os

import numpy as np

import oracle
import precision_quantization_token_gb300 as tk
from bruteforce import decode

SENTINEL_CODE = 0xA5
SENTINEL_WORD = 0x5A5A5A5A
POISON_BF16 = 0x7F00          # 1.7e38: must never be read as input
THREADS = os.cpu_count() or 1

FMT_ID = {"e4m3": oracle.FMT_E4M3, "e2m1": oracle.FMT_E2M1}
MODE_ID = {"fp32": oracle.SCALE_FP32, "pow2": oracle.SCALE_FP32_POW2,
           "ue8m0": oracle.SCALE_UE8M0}
LAYOUT_ID = {"row": oracle.LAYOUT_ROW_MAJOR,
             "transposed": oracle.LAYOUT_TRANSPOSED}


def torch_mod():
    import torch
    return torch


class Case:
    """Buffers for one cast: host input, guard-banded output buffers."""

    def __init__(self, bits, K, group, fmt, mode, layout, swiglu=False,
                 ld_x=None, code_pad=0, scale_pad=0, gain=None, eps=1e-6):
        """gain (BF16 bits [K]) given: the RMSNorm + cast op with that gain
        and eps; swiglu: the fused SwiGLU op; else the plain cast."""
        self.gain = None if gain is None else np.ascontiguousarray(gain, np.uint16)
        self.eps = eps
        self.bits = np.ascontiguousarray(bits, np.uint16)
        self.M = self.bits.shape[0]
        self.K, self.group, self.fmt, self.mode = K, group, fmt, mode
        self.layout, self.swiglu = layout, swiglu
        in_cols = 2 * K if swiglu else K
        assert self.bits.shape[1] == in_cols
        self.ld_x = ld_x or in_cols
        row_bytes = K if fmt == "e4m3" else K // 2
        self.ld_codes = (row_bytes + code_pad + 15) // 16 * 16
        G = K // group
        words = (G + 3) // 4 if mode == "ue8m0" else G
        if layout == "row":
            self.s_rows, self.ld_scales = self.M, words + scale_pad
        else:
            self.s_rows = words
            self.ld_scales = (self.M + 3) // 4 * 4 + 4 * scale_pad
        # host input with a poisoned stride pad
        self.x_host = np.full((self.M, self.ld_x), POISON_BF16, np.uint16)
        self.x_host[:, :in_cols] = self.bits

    def fresh_outputs(self):
        codes = np.full((self.M + 2, self.ld_codes), SENTINEL_CODE, np.uint8)
        scales = np.full((self.s_rows + 2, self.ld_scales), SENTINEL_WORD,
                         np.uint32)
        return codes, scales

    # ---------------------------------------------------------------- GPU
    def run_gpu(self, stream=None, entry=None):
        torch = torch_mod()
        codes, scales = self.fresh_outputs()
        xd = torch.from_numpy(self.x_host.view(np.int16)).cuda()
        cd = torch.from_numpy(codes).cuda()
        sd = torch.from_numpy(scales.view(np.int32)).cuda()
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        if self.gain is not None:
            wd = torch.from_numpy(self.gain.view(np.int16)).cuda()
            tk.tk_rmsnorm_per_token_cast(
                xd.data_ptr(), wd.data_ptr(), self.M, self.K, self.ld_x,
                self.eps, self.group, tk.FMT[self.fmt], tk.SCALE[self.mode],
                tk.LAYOUT[self.layout], cd.data_ptr() + self.ld_codes,
                self.ld_codes, sd.data_ptr() + self.ld_scales * 4,
                self.ld_scales, stream)
            torch.cuda.synchronize()
            return cd.cpu().numpy(), sd.cpu().numpy().view(np.uint32)
        if entry is None:
            entry = (tk.tk_swiglu_per_token_cast if self.swiglu
                     else tk.tk_per_token_cast)
        entry(xd.data_ptr(), self.M, self.K, self.ld_x, self.group,
              tk.FMT[self.fmt], tk.SCALE[self.mode], tk.LAYOUT[self.layout],
              cd.data_ptr() + self.ld_codes, self.ld_codes,
              sd.data_ptr() + self.ld_scales * 4, self.ld_scales, stream)
        torch.cuda.synchronize()
        return cd.cpu().numpy(), sd.cpu().numpy().view(np.uint32)

    # ------------------------------------------------------------- oracle
    def run_oracle(self):
        codes, scales = self.fresh_outputs()
        fn = (oracle.swiglu_per_token_cast if self.swiglu
              else oracle.per_token_cast)
        s_view = scales[1:self.s_rows + 1]
        if self.mode != "ue8m0":
            s_view = s_view.view(np.float32)
        else:
            s_view = s_view.view(np.int32)
        if self.gain is not None:
            oracle.rmsnorm_per_token_cast(
                self.x_host, self.gain, self.K, self.eps, self.group,
                FMT_ID[self.fmt], MODE_ID[self.mode], LAYOUT_ID[self.layout],
                codes=codes[1:self.M + 1], scales=s_view, threads=THREADS)
            return codes, scales
        fn(self.x_host, self.K, self.group, FMT_ID[self.fmt],
           MODE_ID[self.mode], LAYOUT_ID[self.layout],
           codes=codes[1:self.M + 1], scales=s_view, threads=THREADS)
        return codes, scales


def assert_bit_exact(case: Case, gpu=None, ref=None):
    gpu = gpu or case.run_gpu()
    ref = ref or case.run_oracle()
    gc, gs = gpu
    rc, rs = ref
    if not np.array_equal(gc, rc):
        bad = np.argwhere(gc != rc)
        r, c = bad[0]
        raise AssertionError(
            f"codes differ at {bad.shape[0]} bytes; first (row {r - 1}, byte "
            f"{c}): gpu {gc[r, c]:#04x} oracle {rc[r, c]:#04x}")
    if not np.array_equal(gs, rs):
        bad = np.argwhere(gs != rs)
        r, c = bad[0]
        raise AssertionError(
            f"scales differ at {bad.shape[0]} words; first ({r - 1}, {c}): "
            f"gpu {gs[r, c]:#010x} oracle {rs[r, c]:#010x}")


# ------------------------------------------------------- SwiGLU tolerance

def _ordinal(codes, fmt):
    sb = 0x80 if fmt == "e4m3" else 0x8
    c = codes.astype(np.int64)
    mag = c & (sb - 1)
    return np.where(c & sb, -mag, mag)


def _unpack(codes_rows, fmt):
    if fmt == "e4m3":
        return codes_rows
    out = np.empty(codes_rows.shape[:-1] + (codes_rows.shape[-1] * 2,),
                   np.uint8)
    out[..., 0::2] = codes_rows & 0xF
    out[..., 1::2] = codes_rows >> 4
    return out


def _group_scale_values(case: Case, scales_rows):
    """[M, G] float64 scale per group from a scale buffer (guards removed)."""
    M, G = case.M, case.K // case.group
    if case.mode == "ue8m0":
        b = scales_rows.view(np.uint8).reshape(scales_rows.shape[0], -1)
        if case.layout == "row":
            e = b[:M, :G].astype(np.int64)
        else:
            w = b.reshape(scales_rows.shape[0], -1, 4)
            e = np.stack([w[j // 4, :M, j % 4] for j in range(G)],
                         axis=1).astype(np.int64)
        return e
    f = scales_rows.view(np.float32)
    return (f[:M, :G] if case.layout == "row" else f[:G, :M].T)


def check_swiglu(case: Case, gpu=None, ref=None, max_code_frac=1e-4):
    """Tolerance compare of the fused SwiGLU path: fp32 scales within 1 ulp,
    power-of-two scales equal away from 8 ulps of a power of two (see
    check_close)."""
    return check_close(case, gpu, ref, max_code_frac, scale_ulps=1,
                       edge_ulps=8)


def _oracle_values(case: Case):
    K = case.K
    if case.gain is not None:
        return oracle.rmsnorm_values(case.x_host, case.gain, K, case.eps,
                                     threads=THREADS)
    return oracle.swiglu_values(case.x_host[:, :2 * K], K, threads=THREADS)


def check_close(case: Case, gpu=None, ref=None, max_code_frac=1e-4,
                scale_ulps=1, edge_ulps=8, band_ulps=None):
    """Tolerance compare of a fused path whose fp32 values (SwiGLU, RMSNorm)
    may differ from the oracle's by a few ulps.

    Scales: UE8M0 / pow2 equal, except groups whose oracle ratio
    r = max(amax, 1e-4)/fmt_max lies within edge_ulps fp32 ulps of a power
    of two, where a factor-2 difference is allowed (and those groups' codes
    are not compared); fp32 scales within scale_ulps ulps.  Codes: at most
    max_code_frac of the compared elements differ, each by one code step
    (adjacent values on the signed code line).  With band_ulps, every
    differing code must also sit where rounding noise can decide it: the
    oracle's quotient y / s (in double) lies within band_ulps fp32 ulps
    (relative) of the midpoint between the two codes' values.  Guards and
    pads must be untouched.
    """
    gpu = gpu or case.run_gpu()
    ref = ref or case.run_oracle()
    gc, gs = gpu
    rc, rs = ref
    M, K, group = case.M, case.K, case.group
    G = K // group
    row_bytes = K if case.fmt == "e4m3" else K // 2
    # guards / pads untouched: everything outside the written region equal
    assert np.array_equal(gc[0], rc[0]) and np.array_equal(gc[-1], rc[-1])
    assert np.array_equal(gc[:, row_bytes:], rc[:, row_bytes:])
    assert np.array_equal(gs[0], rs[0]) and np.array_equal(gs[-1], rs[-1])

    sg = _group_scale_values(case, gs[1:-1])
    sr = _group_scale_values(case, rs[1:-1])
    fmt_max = 448.0 if case.fmt == "e4m3" else 6.0
    if case.mode == "fp32":
        ug = sg.astype(np.float32).view(np.int32).astype(np.int64)
        ur = sr.astype(np.float32).view(np.int32).astype(np.int64)
        worst = int(np.abs(ug - ur).max(initial=0))
        assert worst <= scale_ulps, f"fp32 scale {worst} ulps off"
        scale_ok = np.ones((M, G), bool)
    else:
        if case.mode == "pow2":
            sg = np.log2(sg.astype(np.float64)).astype(np.int64) + 127
            sr = np.log2(sr.astype(np.float64)).astype(np.int64) + 127
        scale_ok = sg == sr
        if not scale_ok.all():
            y = _oracle_values(case)
            amax = np.abs(y.reshape(M, G, group)).max(axis=2)
            r = np.maximum(amax, np.float32(1e-4)) / np.float32(fmt_max)
            r = r.astype(np.float32)
            p2 = np.exp2(np.round(np.log2(r.astype(np.float64))))
            near = (np.abs(r.astype(np.float64) - p2) <=
                    edge_ulps * np.spacing(r).astype(np.float64))
            bad = ~scale_ok & ~(near & (np.abs(sg - sr) == 1))
            assert not bad.any(), "UE8M0 scale differs away from a 2^k edge"
    codes_g = _unpack(gc[1:-1, :row_bytes], case.fmt).reshape(M, G, group)
    codes_r = _unpack(rc[1:-1, :row_bytes], case.fmt).reshape(M, G, group)
    d = np.abs(_ordinal(codes_g, case.fmt) - _ordinal(codes_r, case.fmt))
    if band_ulps is not None and (d[scale_ok] > 0).any():
        y = _oracle_values(case).reshape(M, G, group).astype(np.float64)
        srv = _group_scale_values(case, rs[1:-1]).astype(np.float64)
        if case.mode == "ue8m0":
            srv = np.exp2(srv - 127)
        q = y / srv[:, :, None]
        sel = (d > 0) & scale_ok[:, :, None]
        vg = decode(codes_g[sel], case.fmt)
        vr = decode(codes_r[sel], case.fmt)
        mid = (vg + vr) / 2
        off = np.abs(q[sel] - mid) / np.maximum(np.abs(mid), 1e-30)
        assert np.all(off <= band_ulps * 2.0 ** -24), (
            f"a code differs away from a rounding midpoint ({off.max():.2e})")
    d = d[scale_ok]
    assert d.max(initial=0) <= 1, "a code differs by more than one step"
    frac = np.count_nonzero(d) / max(1, d.size)
    assert frac <= max_code_frac, f"{frac:.2e} of codes differ"
    return {"code_diff_frac": frac,
            "scale_edge_groups": int((~scale_ok).sum()),
            "max_scale_ulps": (worst if case.mode == "fp32" else 0)}
