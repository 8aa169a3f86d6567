"""Seeded synthetic inputs for the per-token cast (no arithmetic of the cast).

This module is the one piece that both the CUDA path's callers (benchmark,
tests) and the CPU oracle's callers use: it only draws random BF16 matrices
and names the workloads.  It computes no amax, scale or code.

Workloads are the shapes and value mixes the per-token cast is measured on:

  c1   E4M3, 256 x 1024, group 128, fp32 scales, row-major; N(0,1)
  c2   E4M3, 4096 x 7168, group 128, UE8M0 scales packed 4 per int32,
       row-major; N(0,1) with a seeded 0.1% of elements multiplied by 100
  c3a  E4M3, 16384 x 4096, group 32, fp32 scales stored transposed
       [G][M_pad]; N(0,1) times a per-row factor drawn from U(0.01, 10)
  c3b  the same with group 64
  c4   fused SwiGLU: input 8192 x 4096 = [gate | up], output 8192 x 2048,
       E4M3, group 128, UE8M0 packed; N(0,1)
  c5   E2M1, 32768 x 7168, group 16, UE8M0 packed; N(0,1) with a seeded 1%
       of rows all +0 and a disjoint 1% of rows of BF16 denormals (exponent
       field 0, mantissa uniform in 1..127, random sign)
  d2   dequantization of c2's codes and scales to BF16 (4096 x 7168)
  b2   cast-and-cast-back of c2's input (4096 x 7168, E4M3 g128 UE8M0)
  pb2  per-block cast (128 x 128 blocks) of c2's input, E4M3, fp32 scales
  r2   RMSNorm (eps 1e-6, gain 1 + 0.1 N(0,1)) fused with the per-token cast
       of c2's input: E4M3, group 128, UE8M0 packed
  pc2  per-channel cast (one scale per column) of c2's input, E4M3, fp32
  pbd2 / pcd2  dequantization of pb2's / pc2's codes and scales to BF16

Random draws use numpy's PCG64 generator seeded per workload; fp32 values are
rounded to BF16 with round-to-nearest-even on the bit pattern.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_CHUNK = 1 << 24


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int          # channels cast per row (the SwiGLU output width N)
    group: int
    fmt: str        # "e4m3" | "e2m1"
    scale: str      # "fp32" | "pow2" | "ue8m0"
    layout: str     # "row" | "transposed"
    swiglu: bool
    seed: int
    dist: str
    op: str = "cast"   # "cast" | "swiglu" | "dequant" | "cast_back"
    #                  | "block" | "channel" | "rmsnorm"
    #                  | "block_dequant" | "channel_dequant"
    eps: float = 1e-6  # RMSNorm

    @property
    def in_cols(self) -> int:
        return 2 * self.K if self.swiglu else self.K

    @property
    def groups(self) -> int:
        return self.K // self.group

    def algorithmic_bytes(self) -> dict:
        """Bytes read once and written once (padding not counted)."""
        codes = self.M * self.K if self.fmt == "e4m3" else self.M * self.K // 2
        if self.scale == "ue8m0":
            scales = self.M * ((self.groups + 3) // 4) * 4
        else:
            scales = self.M * self.groups * 4
        if self.op == "dequant":
            out = self.M * self.K * 2
            return {"read": codes + scales, "bf16_out": out,
                    "total": codes + scales + out}
        if self.op == "cast_back":
            read = self.M * self.K * 2
            return {"read": read, "bf16_out": read, "total": 2 * read}
        if self.op in ("block", "channel", "block_dequant", "channel_dequant"):
            if self.op.startswith("block"):
                n = -(-self.K // 128)
                rows = -(-self.M // 128)
            else:
                n, rows = self.K, 1
            words = (n + 3) // 4 if self.scale == "ue8m0" else n
            scales = rows * words * 4
            read = self.M * self.K * 2
            if self.op in ("block_dequant", "channel_dequant"):
                return {"read": codes + scales, "bf16_out": read,
                        "total": codes + scales + read}
            return {"read": read, "codes": codes, "scales": scales,
                    "total": read + codes + scales}
        read = self.M * self.in_cols * 2
        if self.op == "rmsnorm":
            read += self.K * 2                      # the gain vector
        return {"read": read, "codes": codes, "scales": scales,
                "total": read + codes + scales}

    def describe(self) -> str:
        if self.op == "block":
            return (f"per_block_cast {self.fmt.upper()} 128x128 blocks "
                    f"{self.scale} {self.M}x{self.K} ({self.dist})")
        if self.op == "channel":
            return (f"per_channel_cast {self.fmt.upper()} {self.scale} "
                    f"{self.M}x{self.K} ({self.dist})")
        if self.op in ("block_dequant", "channel_dequant"):
            kind = "block" if self.op.startswith("block") else "channel"
            return (f"per_{kind}_dequant {self.fmt.upper()} {self.scale} "
                    f"{self.M}x{self.K} -> BF16 ({self.dist})")
        op = {"cast": "per_token_cast", "swiglu": "swiglu_per_token_cast",
              "dequant": "per_token_dequant",
              "cast_back": "per_token_cast_back",
              "rmsnorm": f"rmsnorm(eps {self.eps:g})+per_token_cast"}[self.op]
        shape = (f"{self.M}x{self.in_cols}->{self.M}x{self.K}" if self.swiglu
                 else f"{self.M}x{self.K}")
        return (f"{op} {self.fmt.upper()} g{self.group} {self.scale} "
                f"{self.layout} {shape} ({self.dist})")


WORKLOADS = {
    "c1": Workload("c1", 256, 1024, 128, "e4m3", "fp32", "row", False, 1,
                   "normal"),
    "c2": Workload("c2", 4096, 7168, 128, "e4m3", "ue8m0", "row", False, 2,
                   "normal, 0.1% x100 outliers"),
    "c3a": Workload("c3a", 16384, 4096, 32, "e4m3", "fp32", "transposed",
                    False, 3, "normal x U(0.01,10) per row"),
    "c3b": Workload("c3b", 16384, 4096, 64, "e4m3", "fp32", "transposed",
                    False, 3, "normal x U(0.01,10) per row"),
    "c4": Workload("c4", 8192, 2048, 128, "e4m3", "ue8m0", "row", True, 4,
                   "normal", op="swiglu"),
    "c5": Workload("c5", 32768, 7168, 16, "e2m1", "ue8m0", "row", False, 5,
                   "normal, 1% zero rows, 1% denormal rows"),
    "d2": Workload("d2", 4096, 7168, 128, "e4m3", "ue8m0", "row", False, 2,
                   "normal, 0.1% x100 outliers", op="dequant"),
    "b2": Workload("b2", 4096, 7168, 128, "e4m3", "ue8m0", "row", False, 2,
                   "normal, 0.1% x100 outliers", op="cast_back"),
    "r2": Workload("r2", 4096, 7168, 128, "e4m3", "ue8m0", "row", False, 2,
                   "normal, 0.1% x100 outliers", op="rmsnorm"),
    "pb2": Workload("pb2", 4096, 7168, 128, "e4m3", "fp32", "row", False, 2,
                    "normal, 0.1% x100 outliers", op="block"),
    "pc2": Workload("pc2", 4096, 7168, 4096, "e4m3", "fp32", "row", False, 2,
                    "normal, 0.1% x100 outliers", op="channel"),
    "pbd2": Workload("pbd2", 4096, 7168, 128, "e4m3", "fp32", "row", False, 2,
                     "normal, 0.1% x100 outliers", op="block_dequant"),
    "pcd2": Workload("pcd2", 4096, 7168, 4096, "e4m3", "fp32", "row", False, 2,
                     "normal, 0.1% x100 outliers", op="channel_dequant"),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to BF16 (nearest, ties to even); returns uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    flat_in, flat_out = a.reshape(-1), out.reshape(-1)
    for s in range(0, flat_in.size, _CHUNK):
        u = flat_in[s:s + _CHUNK].view(np.uint32)
        bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
        flat_out[s:s + _CHUNK] = ((u + bias) >> 16).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns to fp32 values."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(
        np.float32)


def _normal_bf16(rng: np.random.Generator, rows: int, cols: int,
                 row_factor: np.ndarray | None = None) -> np.ndarray:
    out = np.empty((rows, cols), np.uint16)
    step = max(1, _CHUNK // cols)
    for r in range(0, rows, step):
        n = min(step, rows - r)
        v = rng.standard_normal((n, cols), dtype=np.float32)
        if row_factor is not None:
            v *= row_factor[r:r + n, None]
        out[r:r + n] = f32_to_bf16_bits(v)
    return out


def make_input(w: Workload, M: int | None = None) -> np.ndarray:
    """BF16 bit patterns [M, in_cols] for a workload (optionally fewer rows:
    the first M rows are drawn the same way, from the same seed)."""
    M = w.M if M is None else M
    rng = np.random.Generator(np.random.PCG64(w.seed))
    cols = w.in_cols
    if w.dist == "normal":
        return _normal_bf16(rng, M, cols)
    if w.dist.startswith("normal, 0.1% x100"):
        x = np.empty((M, cols), np.float32)
        flat = x.reshape(-1)
        for s in range(0, flat.size, _CHUNK):
            n = min(_CHUNK, flat.size - s)
            flat[s:s + n] = rng.standard_normal(n, dtype=np.float32)
        k = max(1, flat.size // 1000)
        idx = rng.choice(flat.size, size=k, replace=False)
        flat[idx] *= np.float32(100.0)
        return f32_to_bf16_bits(x)
    if w.dist.startswith("normal x U(0.01,10)"):
        factor = rng.uniform(0.01, 10.0, size=M).astype(np.float32)
        return _normal_bf16(rng, M, cols, factor)
    if w.dist.startswith("normal, 1% zero rows"):
        perm = rng.permutation(M)
        n1 = max(1, M // 100) if M >= 3 else 0
        zero_rows, den_rows = perm[:n1], perm[n1:2 * n1]
        x = _normal_bf16(rng, M, cols)
        x[zero_rows] = 0
        if den_rows.size:
            mant = rng.integers(1, 128, size=(den_rows.size, cols),
                                dtype=np.uint16)
            sign = rng.integers(0, 2, size=(den_rows.size, cols),
                                dtype=np.uint16) << 15
            x[den_rows] = sign | mant
        return x
    raise ValueError(f"unknown distribution {w.dist!r}")


def make_gain(w: Workload) -> np.ndarray:
    """RMSNorm gain for a workload: 1 + 0.1 N(0, 1) per channel, as BF16
    bits, from a seed of its own (the input's seed + 1000)."""
    rng = np.random.Generator(np.random.PCG64(w.seed + 1000))
    g = 1.0 + 0.1 * rng.standard_normal(w.K, dtype=np.float32)
    return f32_to_bf16_bits(g.astype(np.float32))


def random_bf16(seed: int, rows: int, cols: int, scale: float = 1.0
                ) -> np.ndarray:
    """Small N(0, scale^2) BF16 matrix for parity cases of arbitrary shape."""
    rng = np.random.Generator(np.random.PCG64(seed))
    v = rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(scale)
    return f32_to_bf16_bits(v)
