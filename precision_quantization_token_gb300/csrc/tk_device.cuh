// Device building blocks shared by the cast kernels (sm_103a): mbarrier
// and bulk-copy primitives with bounded waits, BF16 widening, the hardware
// E4M3 / E2M1 conversions and decodes, and the IEEE fp32 scale and quotient
// steps.  Internal to the library; every file that includes it gets its own
// copies (everything here is in an anonymous namespace).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tk_cast.h"

namespace {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s per wait

// Fault codes recorded by a kernel whose wait ran out (OR-ed together).
constexpr unsigned kFaultConsumerWait = 1u;
constexpr unsigned kFaultProducerWait = 2u;
constexpr unsigned kFaultDrain = 4u;

// -------------------------------------------------------- PTX primitives

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
               ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
      ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity to complete, for at most
// kWaitLimitNs, giving up early if another warp has raised `abort_flag`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// Bulk prefetch of global bytes into L2.  A hint: it reads nothing into the
// program's state and orders nothing, so it may run before a dependency wait.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Bulk asynchronous copy global -> shared (this CTA), completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src,
                                          uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// One BF16 element of shared memory, widened to fp32.
__device__ __forceinline__ float lds_bf16(uint32_t addr) {
  uint16_t h;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr));
  return __uint_as_float((uint32_t)h << 16);
}

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds8(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// BF16 element e (a compile-time index after unrolling) of a loaded chunk.
template <int N8>
__device__ __forceinline__ float bf16_at(const uint4 (&r)[N8], int e) {
  const uint4 q = r[e / 8];
  const int w = (e % 8) / 2;
  const uint32_t word = w == 0 ? q.x : w == 1 ? q.y : w == 2 ? q.z : q.w;
  return __uint_as_float((e & 1) ? (word & 0xFFFF0000u) : (word << 16));
}

// ------------------------------------------------------------ conversions

// Four fp32 -> four E4M3 bytes, element 0 in the lowest byte.  In the cvt,
// the first source lands in the upper half of the 16-bit result.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c,
                                               float d) {
  uint32_t out;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(out)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return out;
}

// Eight fp32 -> eight E2M1 nibbles in one word, element 0 in bits 3:0.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* v) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
        "f"(v[6]), "f"(v[7]));
  return out;
}

// Exact decode of codes to fp32 through the hardware f16x2 conversions
// (every E4M3 and E2M1 value is an fp16 value): two E4M3 codes in the low
// 16 bits of `two` (element 0 in the low byte); two E2M1 codes in the low 8
// bits (element 0 in the low nibble).
__device__ __forceinline__ float2 decode_e4m3x2(uint32_t two) {
  uint32_t h;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h) : "r"(two));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ float2 decode_e2m1x2(uint32_t two) {
  uint32_t h;
  asm("{\n\t.reg .b8 c;\n\tcvt.u8.u32 c, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, c;\n\t}" : "=r"(h) : "r"(two));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Sixteen E4M3 codes (one uint4) or E2M1 codes (one uint2) -> fp32 values.
__device__ __forceinline__ void decode16_e4m3(const uint4& c, float (&v)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 lo = decode_e4m3x2(w[i] & 0xFFFFu);
    const float2 hi = decode_e4m3x2(w[i] >> 16);
    v[4 * i + 0] = lo.x;
    v[4 * i + 1] = lo.y;
    v[4 * i + 2] = hi.x;
    v[4 * i + 3] = hi.y;
  }
}

__device__ __forceinline__ void decode16_e2m1(const uint2& c, float (&v)[16]) {
  const uint32_t w[2] = {c.x, c.y};
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 d = decode_e2m1x2((w[i] >> (8 * b)) & 0xFFu);
      v[8 * i + 2 * b] = d.x;
      v[8 * i + 2 * b + 1] = d.y;
    }
}

// Two fp32 -> two BF16 (round to nearest even), element a in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(b), "f"(a));
  return out;
}

// Sixteen values times s (one IEEE fp32 multiply each), stored at dst as
// BF16 (32 bytes) or fp32 (64 bytes).
__device__ __forceinline__ void store_scaled16(uint8_t* dst, const float (&v)[16],
                                               float s, bool as_fp32) {
  float y[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) y[k] = __fmul_rn(v[k], s);
  if (as_fp32) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      d[i] = make_uint4(__float_as_uint(y[4 * i]), __float_as_uint(y[4 * i + 1]),
                        __float_as_uint(y[4 * i + 2]), __float_as_uint(y[4 * i + 3]));
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 2; ++i)
      d[i] = make_uint4(pack_bf16x2(y[8 * i], y[8 * i + 1]), pack_bf16x2(y[8 * i + 2], y[8 * i + 3]),
                        pack_bf16x2(y[8 * i + 4], y[8 * i + 5]), pack_bf16x2(y[8 * i + 6], y[8 * i + 7]));
  }
}

// ------------------------------------------------------------ scale math

struct GroupScale {
  float s;        // the divisor
  float inv;      // 2^-k (power-of-two modes) or RN(1/s) (fp32 mode)
  uint32_t e;     // biased exponent 127 + k (power-of-two modes)
};

template <int FMT, bool POW2>
__device__ __forceinline__ GroupScale group_scale(float amax) {
  constexpr float kMax = FMT == TK_FMT_E4M3 ? 448.0f : 6.0f;
  const float a = fmaxf(amax, 1e-4f);
  GroupScale g;
  if constexpr (POW2) {
    // 2^ceil(log2 RN(a / fmt_max)) without the division.  With
    // a = m * 2^(E-127), m in [1, 2), and fmt_max = 1.75 * 2^8 (E4M3) or
    // 1.5 * 2^2 (E2M1), the exact ratio is (m / 1.75) * 2^(E-135) or
    // (m / 1.5) * 2^(E-129): at most that power of two while m is at most
    // 1.75 (1.5), just above it otherwise, so the biased exponent is E - 8
    // (E - 2) plus one when a's mantissa field exceeds 1.75's (1.5's).
    // Rounding the ratio to fp32 first changes nothing: a ratio above a
    // power of two is more than half an ulp above it (m exceeds 1.75 by a
    // whole ulp of a, over 4/7 of an ulp of the ratio; 2/3 for 1.5).  a is
    // at least 1e-4 and finite, so the exponent lies in [105, 253] and
    // 2^-k is normal.
    constexpr uint32_t kDrop = FMT == TK_FMT_E4M3 ? 8u : 2u;
    constexpr uint32_t kMant = FMT == TK_FMT_E4M3 ? 0x600000u : 0x400000u;
    const uint32_t u = __float_as_uint(a);
    g.e = (u >> 23) - kDrop + ((u & 0x7FFFFFu) > kMant);
    g.s = __uint_as_float(g.e << 23);
    g.inv = __uint_as_float((254u - g.e) << 23);
  } else {
    const float r = __fdiv_rn(a, kMax);
    g.s = r;
    g.inv = __frcp_rn(r);
    g.e = 0;
  }
  return g;
}

// True when every amax within a relative 2^-16 of m gives the same
// power-of-two scale.  By the exponent rule of group_scale the scale only
// changes where the floored amax crosses 1.75 * 2^j (E4M3) or 1.5 * 2^j
// (E2M1), i.e. where its mantissa field passes 0x600000 (0x400000); moving
// by a relative 2^-16 shifts that field by less than 2^8, so a field more
// than 2^8 from the threshold cannot cross it (nor any other crossing
// point, which lies a whole binade or more away).
template <int FMT>
__device__ __forceinline__ bool pow2_settled(float m) {
  constexpr uint32_t kMant = FMT == TK_FMT_E4M3 ? 0x600000u : 0x400000u;
  const uint32_t f = __float_as_uint(fmaxf(m, 1e-4f)) & 0x7FFFFFu;
  return f - kMant + 256u > 512u;           // |f - kMant| > 256 (unsigned wrap)
}

// ------------------------------------------------------- packed pairs
//
// Two-wide forms of the steps above for BF16 input, using the packed fp32
// instructions of sm_100 and later (mul/fma .rn.f32x2: each half is one
// IEEE operation, the same as its scalar form) and the packed BF16 max.
// They give bit-identical results to the scalar steps with half the
// arithmetic instructions.

// Two fp32 values in one 64-bit register, `lo` in the low half.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// Per half, max(|a|, |b|) of two BF16 pairs (exact; the sign bits of the
// result are the XOR of the operands' signs and carry no meaning).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// max |x| over the 8 BF16 values of a 16-byte chunk, still as a BF16 pair.
__device__ __forceinline__ uint32_t bmax_chunk(const uint4& q) {
  return bmax2(bmax2(q.x, q.y), bmax2(q.z, q.w));
}

// The larger magnitude of a BF16 pair from bmax2, as fp32 (exact).
__device__ __forceinline__ float bmax_value(uint32_t m) {
  return fmaxf(__uint_as_float((m << 16) & 0x7FFFFFFFu), __uint_as_float(m & 0x7FFF0000u));
}

// Quotients of the two BF16 values in `w` (element 0 in the low half).
// Power-of-two scales: the exact products x * 2^-k, with inv2 = (2^-k, 2^-k)
// or any per-half pair of such powers.
// fp32 scales: x / s rounded to nearest from the correctly rounded
// reciprocal inv = RN(1/s) and one FMA residual correction (Markstein's
// method), q0 = RN(x * inv), r = RN(q0 * s - x), q = RN(q0 - r * inv); the
// residual is formed as q0 * s - x and subtracted so that x = -0 gives -0.
// The kernels run it on negated operands, with s2 the scales and inv2 the
// negated reciprocals -inv of the two halves, and -x the BF16 pair with both
// sign bits flipped, widened:
//   q0 = RN((-x) * (-inv))        = RN(x * inv), the same sign
//   r  = RN(q0 * s + (-x))        = RN(q0 * s - x)
//   q  = RN(r * (-inv) + q0)      = RN(q0 - r * inv)
// Each line has the same exact operand value and the same sign for every
// zero term, so the negated form is bit-identical, signed zeros included
// (the host proof enumerates every (x, s) pair the casts produce and checks
// that this equals the IEEE quotient, or, below 2^-64, the same code).  The
// sequence is written in PTX so that no compiler rewrite can alter it.
template <bool POW2>
__device__ __forceinline__ void quotient2(uint32_t w, uint64_t s2, uint64_t inv2,
                                          float& q_lo, float& q_hi) {
  if constexpr (POW2) {
    asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 x, q;\n\t"
        "shl.b32 lo, %2, 16;\n\t"
        "and.b32 hi, %2, 0xFFFF0000;\n\t"
        "mov.b64 x, {lo, hi};\n\t"
        "mul.rn.f32x2 q, x, %3;\n\t"
        "mov.b64 {%0, %1}, q;\n\t}"
        : "=f"(q_lo), "=f"(q_hi)
        : "r"(w), "l"(inv2));
  } else {
    asm("{\n\t.reg .b32 n, lo, hi;\n\t.reg .b64 nx, q0, r, q;\n\t"
        "xor.b32 n, %2, 0x80008000;\n\t"
        "shl.b32 lo, n, 16;\n\t"
        "and.b32 hi, n, 0xFFFF0000;\n\t"
        "mov.b64 nx, {lo, hi};\n\t"
        "mul.rn.f32x2 q0, nx, %4;\n\t"
        "fma.rn.f32x2 r, q0, %3, nx;\n\t"
        "fma.rn.f32x2 q, r, %4, q0;\n\t"
        "mov.b64 {%0, %1}, q;\n\t}"
        : "=f"(q_lo), "=f"(q_hi)
        : "r"(w), "l"(s2), "l"(inv2));
  }
}

// Widened pair of the BF16 word w: element 0 in the low half.
__device__ __forceinline__ uint64_t widen_pair(uint32_t w) {
  return pack_f32x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ float lo_of(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_of(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// The larger of |a|, |b| and c (c >= 0), one three-input max.
__device__ __forceinline__ float max_abs2(float c, float a, float b) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(c), "f"(fabsf(a)), "f"(fabsf(b)));
  return d;
}

// Exact products of two BF16 pairs, (a.lo * b.lo, a.hi * b.hi), as an fp32
// pair, straight from the packed halves (mixed-precision fma, sm_100 and
// later).  A product of two BF16 values has at most 16 significant bits, so
// it is exact in fp32 unless it falls below 2^-126; adding -0 keeps every
// value (signed zeros too), and the one rounding is that of the fp32
// multiply of the widened values.
__device__ __forceinline__ uint64_t bmul2(uint32_t a, uint32_t b) {
  uint64_t d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t.reg .f32 lo, hi;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 lo, al, bl, 0f80000000;\n\t"
      "fma.rn.f32.bf16 hi, ah, bh, 0f80000000;\n\t"
      "mov.b64 %0, {lo, hi};\n\t}"
      : "=l"(d) : "r"(a), "r"(b));
  return d;
}

// Sums of squares of a BF16 pair: s0 = RN(a.lo^2 + s0), s1 = RN(a.hi^2 + s1),
// the same single roundings as an fp32 FMA on the widened values.
__device__ __forceinline__ void bsq_acc2(uint32_t a, float& s0, float& s1) {
  asm("{\n\t.reg .b16 al, ah;\n\tmov.b32 {al, ah}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, al, %0;\n\t"
      "fma.rn.f32.bf16 %1, ah, ah, %1;\n\t}"
      : "+f"(s0), "+f"(s1) : "r"(a));
}

// quotient2's reciprocal operand for a scale: 2^-k for power-of-two
// scales, the negated reciprocal for fp32 scales.
template <bool POW2>
__device__ __forceinline__ float quotient2_inv(const GroupScale& g) {
  return POW2 ? g.inv : -g.inv;
}

}  // namespace
