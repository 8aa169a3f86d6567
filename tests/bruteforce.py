"""Independent brute-force references used to pin the oracle.

Nothing here shares code with ``oracle/`` or with the CUDA library.  The
format facts come from the OCP 8-bit floating point specification (E4M3FN:
4 exponent bits with bias 7, 3 mantissa bits, no infinities, the all-ones
pattern is NaN, largest finite 448) and the OCP Microscaling specification
(E2M1: 2 exponent bits with bias 1, 1 mantissa bit, largest 6; UE8M0: an
unsigned biased exponent, value 2^(e-127)).

* ``decode_table`` lists the value of every non-NaN magnitude code.
* ``nearest_code`` picks, for each value, the magnitude code at the smallest
  distance; on an exact tie the code with the even mantissa (even code
  number) wins.  This is a search over decoded values, not bit arithmetic.
* ``rn_f32`` rounds an exact rational to the nearest binary32 (ties to even,
  gradual underflow), written from the IEEE 754 definition with integers.
* ``cast_bruteforce`` casts a tiny row with exact rationals throughout; only
  the IEEE roundings the op prescribes (the fp32 scale, the fp32 quotient)
  are applied, each through ``rn_f32``.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

F32_1E4 = float(np.float32(1e-4))       # the fp32 constant nearest 1e-4
FMT_MAX = {"e4m3": 448.0, "e2m1": 6.0}


def decode_table(fmt: str) -> np.ndarray:
    """Value of each magnitude code 0..(n-1), float64 (exact)."""
    vals = []
    if fmt == "e4m3":
        for c in range(0x7F):             # 0x7F is NaN
            e, m = c >> 3, c & 7
            vals.append(m / 8 * 2.0 ** -6 if e == 0 else
                        (1 + m / 8) * 2.0 ** (e - 7))
    else:
        for c in range(8):
            e, m = c >> 1, c & 1
            vals.append(m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
    return np.array(vals, dtype=np.float64)


def sign_bit(fmt: str) -> int:
    return 0x80 if fmt == "e4m3" else 0x8


def decode(codes: np.ndarray, fmt: str) -> np.ndarray:
    """Signed value of each code (float64)."""
    table = decode_table(fmt)
    sb = sign_bit(fmt)
    codes = np.asarray(codes).astype(np.int64)
    mag = table[codes & (sb - 1)]
    return np.where(codes & sb, -mag, mag)


def nearest_code(q: np.ndarray, fmt: str) -> np.ndarray:
    """Saturate to +-fmt_max, then the nearest code, ties to even code."""
    q = np.asarray(q, dtype=np.float32).astype(np.float64)
    table = decode_table(fmt)                 # increasing
    neg = np.signbit(q)
    a = np.minimum(np.abs(q), FMT_MAX[fmt])
    hi = np.searchsorted(table, a, side="left")  # first table >= a
    hi = np.clip(hi, 0, table.size - 1)
    lo = np.clip(hi - 1, 0, table.size - 1)
    d_hi = np.abs(table[hi] - a)
    d_lo = np.abs(a - table[lo])
    pick = np.where(d_lo < d_hi, lo,
                    np.where(d_hi < d_lo, hi,
                             np.where(lo % 2 == 0, lo, hi)))
    return (pick | np.where(neg, sign_bit(fmt), 0)).astype(np.uint8)


def rn_f32(x: Fraction) -> float:
    """Round a rational to the nearest IEEE binary32 value, ties to even."""
    if x == 0:
        return 0.0
    neg = x < 0
    a = -x if neg else x
    # e = floor(log2(a))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum_exp = max(e, -126) - 23           # ulp exponent (gradual underflow)
    scaled = a / Fraction(2) ** quantum_exp
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = float(Fraction(n) * Fraction(2) ** quantum_exp)
    if val > float(np.finfo(np.float32).max):
        val = float("inf")
    return -val if neg else val


def pow2_ceil_exponent(x: Fraction) -> int:
    """Smallest k with 2^k >= x (x > 0), by exact comparison."""
    k = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** k < x:
        k += 1
    while Fraction(2) ** (k - 1) >= x:
        k -= 1
    return k


def scale_bruteforce(amax: float, fmt: str, mode: str):
    """(scale, ue8m0 byte or None) with exact rationals.

    fp32 mode: the fp32 quotient of the floored amax by the format maximum.
    pow2 / ue8m0: the smallest power of two >= the exact quotient.
    """
    a = max(amax, F32_1E4)
    ratio = Fraction(a) / Fraction(FMT_MAX[fmt])
    if mode == "fp32":
        return rn_f32(ratio), None
    k = pow2_ceil_exponent(ratio)
    return float(Fraction(2) ** k), k + 127


def cast_bruteforce(row, group: int, fmt: str, mode: str):
    """Tiny-row cast with exact arithmetic: returns (codes list, scales list).

    ``row`` holds fp32-representable Python floats.  Codes are unpacked (one
    per element, sign included); scales are floats (fp32/pow2) or UE8M0 bytes.
    """
    codes, scales = [], []
    for j in range(0, len(row), group):
        grp = row[j:j + group]
        amax = max(abs(v) for v in grp)
        s, e = scale_bruteforce(amax, fmt, mode)
        scales.append(e if mode == "ue8m0" else s)
        q = [rn_f32(Fraction(v) / Fraction(s)) if v != 0 else
             (-0.0 if np.signbit(v) else 0.0) for v in grp]
        codes.extend(int(c) for c in nearest_code(np.array(q, np.float32), fmt))
    return codes, scales
