/*
 * Plain CPU oracle for the per-token, group-wise activation cast
 * (BF16 -> FP8 E4M3 / FP4 E2M1, with fused SwiGLU as a variant).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it follows:
 *  - TileKernels README (pypi tile-kernels 2.0.0), section "Features": the
 *    quantization family offers per-token FP8/FP4 casting with fused
 *    SwiGLU+quantization.
 *  - aiwiki "TileKernels", section "Quantization": the per-token cast takes
 *    scale-factor groups of 16, 32, 64 or 128 channels, optional
 *    power-of-two rounding of the scale and packed UE8M0 scale factors, and
 *    per-token scales "in DeepGEMM's layout" (transposed, M padded).
 *  - The pages give no formula.  The steps below are the op's plain
 *    definition: per group amax, amax floored at 1e-4, scale = amax/fmt_max
 *    in IEEE fp32 (optionally rounded up to 2^k), codes = RNE(sat(x/scale)).
 *  - Number formats: OCP 8-bit floating point spec (E4M3FN: bias 7,
 *    no infinities, max normal 448, subnormal step 2^-9) and OCP
 *    Microscaling spec (E2M1: bias 1, values 0,0.5,1,1.5,2,3,4,6; UE8M0:
 *    unsigned 8-bit exponent, value 2^(e-127)).
 *
 * Every step is written literally, one element at a time, in IEEE fp32
 * (compiled with -ffp-contract=off and without fast-math) except the
 * SwiGLU product, which is formed in double and rounded once to fp32.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_NONFINITE 2

#define OR_FMT_E4M3 0
#define OR_FMT_E2M1 1

#define OR_SCALE_FP32 0
#define OR_SCALE_FP32_POW2 1
#define OR_SCALE_UE8M0 2

#define OR_LAYOUT_ROW_MAJOR 0
#define OR_LAYOUT_TRANSPOSED 1

/* ---------------------------------------------------------------- helpers */

/* BF16 is the upper half of an IEEE binary32: widening is exact. */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t float_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float format_max(int fmt)
{
    return fmt == OR_FMT_E4M3 ? 448.0f : 6.0f;
}

/* ------------------------------------------------------ E4M3FN (OCP FP8) */

/*
 * Magnitude code (7 bits: 4 exponent bits, bias 7, then 3 mantissa bits) of
 * a finite v with 0 <= v <= 448, rounded to nearest, ties to even mantissa.
 * Normal numbers (v >= 2^-6) keep the top 3 fp32 mantissa bits; below 2^-6
 * the format is fixed-point with step 2^-9.
 */
static unsigned e4m3_magnitude(float v)
{
    uint32_t u = float_bits(v);
    int biased = (int)(u >> 23);          /* sign bit is 0 here */
    uint32_t mant = u & 0x7FFFFFu;
    if (biased >= 127 - 6) {
        uint32_t keep = mant >> 20;        /* 3 kept mantissa bits */
        uint32_t dropped = mant & 0xFFFFFu; /* 20 dropped bits */
        int e = biased - 127 + 7;          /* E4M3 biased exponent, >= 1 */
        if (dropped > 0x80000u || (dropped == 0x80000u && (keep & 1u)))
            keep += 1;
        if (keep == 8) {                   /* mantissa overflow: next binade */
            keep = 0;
            e += 1;
        }
        return ((unsigned)e << 3) | keep;
    }
    /* Subnormal range: v = m * 2^-9 with m in [0, 8).  Scaling by 2^9 is
     * exact, and so is splitting t into integer and fractional parts. */
    float t = v * 512.0f;
    unsigned m = (unsigned)t;
    float frac = t - (float)m;
    if (frac > 0.5f || (frac == 0.5f && (m & 1u)))
        m += 1;
    return m; /* m == 8 is exponent 1, mantissa 0: the smallest normal */
}

/* Saturate to +-448, then round to nearest even; the sign of q (including
 * the sign of a zero or of a value that rounds to zero) is kept. */
static uint8_t e4m3_encode(float q)
{
    unsigned sign = signbit(q) ? 0x80u : 0u;
    float a = fabsf(q);
    if (a > 448.0f)
        a = 448.0f;
    return (uint8_t)(sign | e4m3_magnitude(a));
}

/* ------------------------------------------------------- E2M1 (OCP MX FP4) */

/*
 * Magnitude code (3 bits: 2 exponent bits, bias 1, then 1 mantissa bit) of a
 * finite v with 0 <= v <= 6, rounded to nearest, ties to even mantissa.
 * Normal numbers are v >= 1; below 1 the step is 0.5.
 */
static unsigned e2m1_magnitude(float v)
{
    uint32_t u = float_bits(v);
    int biased = (int)(u >> 23);
    uint32_t mant = u & 0x7FFFFFu;
    if (biased >= 127) {
        uint32_t keep = mant >> 22;         /* 1 kept mantissa bit */
        uint32_t dropped = mant & 0x3FFFFFu; /* 22 dropped bits */
        int e = biased - 127 + 1;
        if (dropped > 0x200000u || (dropped == 0x200000u && (keep & 1u)))
            keep += 1;
        if (keep == 2) {
            keep = 0;
            e += 1;
        }
        return ((unsigned)e << 1) | keep;
    }
    float t = v * 2.0f;
    unsigned m = (unsigned)t;
    float frac = t - (float)m;
    if (frac > 0.5f || (frac == 0.5f && (m & 1u)))
        m += 1;
    return m; /* 2 is exponent 1, mantissa 0: the value 1.0 */
}

static uint8_t e2m1_encode(float q)
{
    unsigned sign = signbit(q) ? 0x8u : 0u;
    float a = fabsf(q);
    if (a > 6.0f)
        a = 6.0f;
    return (uint8_t)(sign | e2m1_magnitude(a));
}

/* ------------------------------------------------------------ group scale */

typedef struct {
    float s;      /* the scale the codes are divided by */
    float r;      /* fp32 ratio max(amax, 1e-4) / fmt_max */
    int ue8m0;    /* biased exponent of s when s is a power of two */
} group_scale;

/*
 * amax floored at 1e-4 (the fp32 constant nearest 1e-4), ratio to the
 * format maximum in one IEEE fp32 division.  In the power-of-two modes the
 * scale is the smallest 2^k that is >= the ratio; frexpf splits the ratio
 * as f * 2^E with f in [0.5, 1), so the ratio is itself 2^(E-1) exactly
 * when f == 0.5, and lies strictly between 2^(E-1) and 2^E otherwise.
 */
static group_scale compute_scale(float amax, int fmt, int mode)
{
    group_scale g;
    float a = amax > 1e-4f ? amax : 1e-4f;
    g.r = a / format_max(fmt);
    g.s = g.r;
    g.ue8m0 = -1;
    if (mode != OR_SCALE_FP32) {
        int E;
        float f = frexpf(g.r, &E);
        int k = (f == 0.5f) ? E - 1 : E;
        g.s = ldexpf(1.0f, k);
        g.ue8m0 = k + 127;
    }
    return g;
}

/* ------------------------------------------------------------- row cast */

/*
 * Casts one row of K fp32 values (already exact widenings of BF16, or the
 * fp32 SwiGLU product) in groups of `group` channels.
 *   codes_row : E4M3 -> K bytes; E2M1 -> K/2 bytes, element 2i in the low
 *               nibble of byte i and element 2i+1 in the high nibble.
 *   scales    : base of the whole scale tensor; row m's entries are written
 *               according to mode and layout (see the scale writers below).
 */
static int cast_row(const float *y, int64_t K, int group, int fmt, int mode,
                    int layout, int64_t m, uint8_t *codes_row, void *scales,
                    int64_t ld_scales)
{
    int64_t G = K / group;
    for (int64_t j = 0; j < G; ++j) {
        const float *yg = y + j * group;
        float amax = 0.0f;
        for (int k = 0; k < group; ++k) {
            if (!isfinite(yg[k]))
                return OR_NONFINITE;
            float a = fabsf(yg[k]);
            if (a > amax)
                amax = a;
        }
        group_scale sc = compute_scale(amax, fmt, mode);

        for (int k = 0; k < group; ++k) {
            float q = yg[k] / sc.s;
            int64_t col = j * group + k;
            if (fmt == OR_FMT_E4M3) {
                codes_row[col] = e4m3_encode(q);
            } else {
                uint8_t c = e2m1_encode(q);
                uint8_t *byte = &codes_row[col / 2];
                if ((col & 1) == 0)
                    *byte = (uint8_t)((*byte & 0xF0u) | c);
                else
                    *byte = (uint8_t)((*byte & 0x0Fu) | (c << 4));
            }
        }

        if (mode == OR_SCALE_UE8M0) {
            /* Four exponent bytes per int32, group 4w+b in byte b of word w
             * (little-endian), i.e. byte offset w*4+b inside the word row or
             * column. */
            int64_t w = j / 4, b = j % 4;
            uint8_t *base = (uint8_t *)scales;
            int64_t word = layout == OR_LAYOUT_ROW_MAJOR ? m * ld_scales + w
                                                         : w * ld_scales + m;
            base[word * 4 + b] = (uint8_t)sc.ue8m0;
        } else {
            float *base = (float *)scales;
            if (layout == OR_LAYOUT_ROW_MAJOR)
                base[m * ld_scales + j] = sc.s;
            else
                base[j * ld_scales + m] = sc.s;
        }
    }
    if (mode == OR_SCALE_UE8M0 && (G % 4) != 0) {
        /* Unused bytes of the last, partly filled word are zero. */
        uint8_t *base = (uint8_t *)scales;
        int64_t w = G / 4;
        int64_t word = layout == OR_LAYOUT_ROW_MAJOR ? m * ld_scales + w
                                                     : w * ld_scales + m;
        for (int64_t b = G % 4; b < 4; ++b)
            base[word * 4 + b] = 0;
    }
    return OR_OK;
}

static int check_common(int64_t K, int group, int fmt, int mode, int layout)
{
    if (K <= 0 || (group != 16 && group != 32 && group != 64 && group != 128))
        return OR_BAD_ARG;
    if (K % group != 0)
        return OR_BAD_ARG;
    if (fmt != OR_FMT_E4M3 && fmt != OR_FMT_E2M1)
        return OR_BAD_ARG;
    if (mode < OR_SCALE_FP32 || mode > OR_SCALE_UE8M0)
        return OR_BAD_ARG;
    if (layout != OR_LAYOUT_ROW_MAJOR && layout != OR_LAYOUT_TRANSPOSED)
        return OR_BAD_ARG;
    return OR_OK;
}

/* ---------------------------------------------------------- public entry */

/*
 * Per-token cast of rows [m_begin, m_end) of a BF16 matrix.
 *   x        : BF16 bit patterns, row m at x + m*ld_x, K values.
 *   codes    : row m at codes + m*ld_codes (bytes).
 *   scales   : fp32 (modes 0, 1) or packed UE8M0 int32 words (mode 2);
 *              row-major [M][ld_scales] or transposed [G or ceil(G/4)][ld_scales].
 * Returns 0, or OR_NONFINITE if a row holds a NaN or an infinity (outside
 * the op's contract), or OR_BAD_ARG.
 */
int oracle_per_token_cast(const uint16_t *x, int64_t m_begin, int64_t m_end,
                          int64_t K, int64_t ld_x, int group, int fmt, int mode,
                          int layout, uint8_t *codes, int64_t ld_codes,
                          void *scales, int64_t ld_scales)
{
    int rc = check_common(K, group, fmt, mode, layout);
    if (rc != OR_OK)
        return rc;
    float *row = (float *)malloc((size_t)K * sizeof(float));
    if (!row)
        return OR_BAD_ARG;
    for (int64_t m = m_begin; m < m_end && rc == OR_OK; ++m) {
        const uint16_t *xr = x + m * ld_x;
        for (int64_t k = 0; k < K; ++k)
            row[k] = bf16_bits_to_float(xr[k]);
        rc = cast_row(row, K, group, fmt, mode, layout, m,
                      codes + m * ld_codes, scales, ld_scales);
    }
    free(row);
    return rc;
}

/*
 * SwiGLU value for one (gate, up) pair: gate * up / (1 + e^-gate), formed
 * in double and rounded once to fp32.  silu(v) = v * sigmoid(v).
 */
float oracle_swiglu_value(float gate, float up)
{
    double g = (double)gate, u = (double)up;
    return (float)(g * u / (1.0 + exp(-g)));
}

/*
 * Fused SwiGLU + per-token cast of rows [m_begin, m_end).  Row m of x holds
 * 2N BF16 values: gate in columns [0, N), up in columns [N, 2N).  The fp32
 * product row of N values is cast exactly as oracle_per_token_cast casts a
 * row of K = N values.
 */
int oracle_swiglu_per_token_cast(const uint16_t *x, int64_t m_begin,
                                 int64_t m_end, int64_t N, int64_t ld_x,
                                 int group, int fmt, int mode, int layout,
                                 uint8_t *codes, int64_t ld_codes, void *scales,
                                 int64_t ld_scales)
{
    int rc = check_common(N, group, fmt, mode, layout);
    if (rc != OR_OK)
        return rc;
    float *row = (float *)malloc((size_t)N * sizeof(float));
    if (!row)
        return OR_BAD_ARG;
    for (int64_t m = m_begin; m < m_end && rc == OR_OK; ++m) {
        const uint16_t *xr = x + m * ld_x;
        for (int64_t k = 0; k < N; ++k)
            row[k] = oracle_swiglu_value(bf16_bits_to_float(xr[k]),
                                         bf16_bits_to_float(xr[N + k]));
        rc = cast_row(row, N, group, fmt, mode, layout, m,
                      codes + m * ld_codes, scales, ld_scales);
    }
    free(row);
    return rc;
}

/* The fp32 SwiGLU product rows alone (no cast): y row m at y + m*ld_y. */
void oracle_swiglu_values(const uint16_t *x, int64_t m_begin, int64_t m_end,
                          int64_t N, int64_t ld_x, float *y, int64_t ld_y)
{
    for (int64_t m = m_begin; m < m_end; ++m) {
        const uint16_t *xr = x + m * ld_x;
        for (int64_t k = 0; k < N; ++k)
            y[m * ld_y + k] = oracle_swiglu_value(bf16_bits_to_float(xr[k]),
                                                  bf16_bits_to_float(xr[N + k]));
    }
}

/* ------------------------------------------------ dequantization (decode) */

/*
 * Value of an E4M3FN code (OCP 8-bit floating point): sign | exponent e
 * (bias 7) | mantissa m (3 bits); e == 0 is subnormal, m * 2^-9.  The NaN
 * pattern S.1111.111 is never produced by the cast; it decodes to NaN.
 */
static float e4m3_decode(uint8_t c)
{
    int e = (c >> 3) & 0xF, m = c & 7;
    float mag;
    if (e == 15 && m == 7)
        mag = NAN;
    else if (e == 0)
        mag = ldexpf((float)m, -9);
    else
        mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return (c & 0x80) ? -mag : mag;
}

/* Value of an E2M1 code (OCP MX): sign | exponent e (bias 1) | mantissa m
 * (1 bit); e == 0 is subnormal, m * 0.5. */
static float e2m1_decode(uint8_t c)
{
    int e = (c >> 1) & 3, m = c & 1;
    float mag = e == 0 ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
    return (c & 0x8) ? -mag : mag;
}

/* fp32 -> BF16 bits, round to nearest, ties to even (NaN kept quiet). */
static uint16_t float_to_bf16_bits(float f)
{
    uint32_t u = float_bits(f);
    if (isnan(f))
        return (uint16_t)((u >> 16) | 0x40);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1;                       /* carries into the exponent too */
    return (uint16_t)upper;
}

/* Scale of group j of row m read back from a scale tensor written by the
 * cast (fp32 value, or 2^(byte-127) for packed UE8M0). */
static float read_scale(const void *scales, int64_t ld_scales, int mode,
                        int layout, int64_t m, int64_t j)
{
    if (mode == OR_SCALE_UE8M0) {
        const uint8_t *base = (const uint8_t *)scales;
        int64_t w = j / 4, b = j % 4;
        int64_t word = layout == OR_LAYOUT_ROW_MAJOR ? m * ld_scales + w
                                                     : w * ld_scales + m;
        return ldexpf(1.0f, (int)base[word * 4 + b] - 127);
    }
    const float *base = (const float *)scales;
    return layout == OR_LAYOUT_ROW_MAJOR ? base[m * ld_scales + j]
                                         : base[j * ld_scales + m];
}

/*
 * Per-token dequantization of rows [m_begin, m_end): y = code value * scale,
 * one fp32 multiply per element, written as fp32 (out_fp32 != 0) or rounded
 * to BF16 (nearest even).  codes/scales are laid out as the cast writes them.
 * y row m at y + m * ld_y (elements of the output type).
 */
int oracle_per_token_dequant(const uint8_t *codes, int64_t ld_codes,
                             const void *scales, int64_t ld_scales,
                             int64_t m_begin, int64_t m_end, int64_t K,
                             int group, int fmt, int mode, int layout,
                             int out_fp32, void *y, int64_t ld_y)
{
    int rc = check_common(K, group, fmt, mode, layout);
    if (rc != OR_OK)
        return rc;
    for (int64_t m = m_begin; m < m_end; ++m) {
        const uint8_t *cr = codes + m * ld_codes;
        for (int64_t k = 0; k < K; ++k) {
            float v;
            if (fmt == OR_FMT_E4M3) {
                v = e4m3_decode(cr[k]);
            } else {
                uint8_t byte = cr[k / 2];
                v = e2m1_decode((uint8_t)((k & 1) ? byte >> 4 : byte & 0xF));
            }
            float s = read_scale(scales, ld_scales, mode, layout, m, k / group);
            float prod = v * s;
            if (out_fp32)
                ((float *)y)[m * ld_y + k] = prod;
            else
                ((uint16_t *)y)[m * ld_y + k] = float_to_bf16_bits(prod);
        }
    }
    return OR_OK;
}

/*
 * Per-token cast-and-cast-back (quantisation round trip) of rows
 * [m_begin, m_end): each row is cast exactly as oracle_per_token_cast casts
 * it, then dequantized as oracle_per_token_dequant does, into BF16 y.
 */
int oracle_per_token_cast_back(const uint16_t *x, int64_t m_begin,
                               int64_t m_end, int64_t K, int64_t ld_x,
                               int group, int fmt, int mode, uint16_t *y,
                               int64_t ld_y)
{
    int rc = check_common(K, group, fmt, mode, OR_LAYOUT_ROW_MAJOR);
    if (rc != OR_OK)
        return rc;
    int64_t G = K / group;
    int64_t words = mode == OR_SCALE_UE8M0 ? (G + 3) / 4 : G;
    float *row = (float *)malloc((size_t)K * sizeof(float));
    uint8_t *codes = (uint8_t *)calloc((size_t)K, 1);
    uint32_t *sc = (uint32_t *)calloc((size_t)words, sizeof(uint32_t));
    if (!row || !codes || !sc) {
        free(row);
        free(codes);
        free(sc);
        return OR_BAD_ARG;
    }
    for (int64_t m = m_begin; m < m_end && rc == OR_OK; ++m) {
        const uint16_t *xr = x + m * ld_x;
        for (int64_t k = 0; k < K; ++k)
            row[k] = bf16_bits_to_float(xr[k]);
        /* one-row scratch: row index 0, row-major scales */
        rc = cast_row(row, K, group, fmt, mode, OR_LAYOUT_ROW_MAJOR, 0, codes,
                      sc, words);
        if (rc == OR_OK)
            rc = oracle_per_token_dequant(codes, 0, sc, words, 0, 1, K,
                                          group, fmt, mode,
                                          OR_LAYOUT_ROW_MAJOR, 0,
                                          y + m * ld_y, 0);
    }
    free(row);
    free(codes);
    free(sc);
    return rc;
}

/* ------------------------------------------------- RMSNorm + per-token cast */

/*
 * aiwiki "TileKernels", section "Version 2.0.0": the library added RMSNorm
 * forward and backward "with an optional fused FP8 cast".  The pages do not
 * define RMSNorm; this follows its published definition (Zhang and Sennrich,
 * "Root Mean Square Layer Normalization", 2019), with a learned gain w per
 * channel and eps added to the mean square:
 *   y_k = w_k * x_k / sqrt(eps + (1/K) * sum_j x_j^2)
 * Formed in double (every BF16 square and product is exact there and the
 * sum of K <= 2^28 positive terms is within a few double ulps) and rounded
 * once to fp32; the fused cast then casts y exactly as cast_row casts an
 * fp32 row (no BF16 intermediate).  A row of zeros with eps = 0 has no
 * value (0/0): the cast returns OR_NONFINITE for it.
 */
void oracle_rmsnorm_values(const uint16_t *x, const uint16_t *w,
                           int64_t m_begin, int64_t m_end, int64_t K,
                           int64_t ld_x, float eps, float *y, int64_t ld_y)
{
    for (int64_t m = m_begin; m < m_end; ++m) {
        const uint16_t *xr = x + m * ld_x;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = (double)bf16_bits_to_float(xr[k]);
            ss += v * v;
        }
        double rstd = 1.0 / sqrt((double)eps + ss / (double)K);
        for (int64_t k = 0; k < K; ++k)
            y[m * ld_y + k] = (float)((double)bf16_bits_to_float(w[k]) *
                                      (double)bf16_bits_to_float(xr[k]) *
                                      rstd);
    }
}

int oracle_rmsnorm_per_token_cast(const uint16_t *x, const uint16_t *w,
                                  int64_t m_begin, int64_t m_end, int64_t K,
                                  int64_t ld_x, float eps, int group, int fmt,
                                  int mode, int layout, uint8_t *codes,
                                  int64_t ld_codes, void *scales,
                                  int64_t ld_scales)
{
    int rc = check_common(K, group, fmt, mode, layout);
    if (rc != OR_OK)
        return rc;
    if (!(eps >= 0.0f) || !isfinite(eps))
        return OR_BAD_ARG;
    float *row = (float *)malloc((size_t)K * sizeof(float));
    if (!row)
        return OR_BAD_ARG;
    for (int64_t m = m_begin; m < m_end && rc == OR_OK; ++m) {
        oracle_rmsnorm_values(x + m * ld_x, w, 0, 1, K, ld_x, eps, row, K);
        rc = cast_row(row, K, group, fmt, mode, layout, m,
                      codes + m * ld_codes, scales, ld_scales);
    }
    free(row);
    return rc;
}

/* ------------------------------------------ per-block and per-channel cast */

/*
 * TileKernels README (pypi tile-kernels 2.0.0), section "Features", and the
 * hysenlabs page "TileKernels, TileLang kernels for MoE routing and
 * low-precision quantization", section "Seven kernel families, from MoE
 * routing to Sinkhorn normalisation": besides the per-token cast the
 * library casts per block and per channel.  The pages name these and nothing more; the
 * steps are the per-token ones with a different set of elements sharing a
 * scale:
 *   per block   : a square block of `block` rows x `block` channels (the
 *                 library uses 128 x 128; the last block row and block
 *                 column may be partial);
 *   per channel : one channel (column) over all M rows.
 * The amax, floor, scale and code steps are compute_scale and the
 * encoders above, unchanged.
 */

/* One code into a row of codes (E2M1: element 2i in the low nibble of byte
 * i, element 2i+1 in the high nibble). */
static void put_code(uint8_t *codes_row, int64_t col, int fmt, float q)
{
    if (fmt == OR_FMT_E4M3) {
        codes_row[col] = e4m3_encode(q);
        return;
    }
    uint8_t c = e2m1_encode(q);
    uint8_t *byte = &codes_row[col / 2];
    if (col % 2 == 0)
        *byte = (uint8_t)((*byte & 0xF0u) | c);
    else
        *byte = (uint8_t)((*byte & 0x0Fu) | (c << 4));
}

/* Entry i of a vector of scales: fp32 word i, or, for packed UE8M0, byte
 * i % 4 of word i / 4 (little-endian: byte i of the vector's bytes). */
static void put_scale(void *vec, int64_t i, int mode, group_scale sc)
{
    if (mode == OR_SCALE_UE8M0)
        ((uint8_t *)vec)[i] = (uint8_t)sc.ue8m0;
    else
        ((float *)vec)[i] = sc.s;
}

/* Unused bytes of the last, partly filled packed UE8M0 word are zero. */
static void zero_word_tail(void *vec, int64_t n)
{
    for (int64_t i = n; i % 4 != 0; ++i)
        ((uint8_t *)vec)[i] = 0;
}

static int check_tile_args(int64_t M, int64_t K, int fmt, int mode)
{
    if (M < 0 || K <= 0)
        return OR_BAD_ARG;
    if (fmt != OR_FMT_E4M3 && fmt != OR_FMT_E2M1)
        return OR_BAD_ARG;
    if (fmt == OR_FMT_E2M1 && K % 2 != 0)
        return OR_BAD_ARG;
    if (mode < OR_SCALE_FP32 || mode > OR_SCALE_UE8M0)
        return OR_BAD_ARG;
    return OR_OK;
}

/*
 * Per-block cast of block rows [rb_begin, rb_end).
 *   x      : BF16 bit patterns, row m at x + m*ld_x, K values.
 *   codes  : row m at codes + m*ld_codes (bytes), as the per-token cast.
 *   scales : 4-byte words, block row rb at scales + rb*ld_scales words;
 *            block column j is fp32 word j, or byte j of the row's packed
 *            UE8M0 words (unused bytes of the last word zero).
 */
int oracle_per_block_cast(const uint16_t *x, int64_t M, int64_t K,
                          int64_t ld_x, int block, int64_t rb_begin,
                          int64_t rb_end, int fmt, int mode, uint8_t *codes,
                          int64_t ld_codes, void *scales, int64_t ld_scales)
{
    if (block != 16 && block != 32 && block != 64 && block != 128)
        return OR_BAD_ARG;
    int rc = check_tile_args(M, K, fmt, mode);
    if (rc != OR_OK)
        return rc;
    int64_t n_cb = (K + block - 1) / block;
    for (int64_t rb = rb_begin; rb < rb_end; ++rb) {
        int64_t r0 = rb * block;
        int64_t r1 = r0 + block < M ? r0 + block : M;
        uint8_t *srow = (uint8_t *)scales + rb * ld_scales * 4;
        for (int64_t cb = 0; cb < n_cb; ++cb) {
            int64_t c0 = cb * block;
            int64_t c1 = c0 + block < K ? c0 + block : K;
            float bmax = 0.0f;
            for (int64_t r = r0; r < r1; ++r) {
                for (int64_t c = c0; c < c1; ++c) {
                    float v = bf16_bits_to_float(x[r * ld_x + c]);
                    if (!isfinite(v))
                        return OR_NONFINITE;
                    if (fabsf(v) > bmax)
                        bmax = fabsf(v);
                }
            }
            group_scale sc = compute_scale(bmax, fmt, mode);
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = c0; c < c1; ++c)
                    put_code(codes + r * ld_codes, c, fmt,
                             bf16_bits_to_float(x[r * ld_x + c]) / sc.s);
            put_scale(srow, cb, mode, sc);
        }
        if (mode == OR_SCALE_UE8M0)
            zero_word_tail(srow, n_cb);
    }
    return OR_OK;
}

/*
 * Per-channel cast of channels [k_begin, k_end) over all M rows.
 *   scales : a vector, channel k at fp32 word k or byte k of the packed
 *            UE8M0 words (the unused bytes of the last word are zeroed by
 *            the call whose range ends at K).
 * Callers splitting the channels keep k_begin a multiple of 4 (two E2M1
 * codes share a byte; four UE8M0 bytes share a word).  M == 0 writes
 * nothing: there is no element to take a scale from.
 */
int oracle_per_channel_cast(const uint16_t *x, int64_t M, int64_t K,
                            int64_t ld_x, int64_t k_begin, int64_t k_end,
                            int fmt, int mode, uint8_t *codes,
                            int64_t ld_codes, void *scales)
{
    int rc = check_tile_args(M, K, fmt, mode);
    if (rc != OR_OK)
        return rc;
    if (M == 0)
        return OR_OK;
    for (int64_t k = k_begin; k < k_end; ++k) {
        float cmax = 0.0f;
        for (int64_t m = 0; m < M; ++m) {
            float v = bf16_bits_to_float(x[m * ld_x + k]);
            if (!isfinite(v))
                return OR_NONFINITE;
            if (fabsf(v) > cmax)
                cmax = fabsf(v);
        }
        group_scale sc = compute_scale(cmax, fmt, mode);
        for (int64_t m = 0; m < M; ++m)
            put_code(codes + m * ld_codes, k, fmt,
                     bf16_bits_to_float(x[m * ld_x + k]) / sc.s);
        put_scale(scales, k, mode, sc);
    }
    if (mode == OR_SCALE_UE8M0 && k_end == K)
        zero_word_tail(scales, K);
    return OR_OK;
}

/* --------------------------------- per-block and per-channel dequantization */

/*
 * TileKernels README, "Features": the per-block and per-channel casts come
 * with dequantization.  Its element step is the per-token one: the code's
 * exact value times the scale of the code's block (or channel), one IEEE
 * fp32 multiply, stored as fp32 or rounded to BF16 (nearest even); codes
 * and scales are laid out as oracle_per_block_cast / oracle_per_channel_cast
 * write them.  Rows [m_begin, m_end) are processed; y row m at y + m*ld_y
 * elements of the output type.
 */
static float code_value(const uint8_t *code_row, int64_t k, int fmt)
{
    if (fmt == OR_FMT_E4M3)
        return e4m3_decode(code_row[k]);
    uint8_t byte = code_row[k / 2];
    return e2m1_decode((uint8_t)((k & 1) ? byte >> 4 : byte & 0xF));
}

static void put_output(void *y, int64_t at, int out_fp32, float value)
{
    if (out_fp32)
        ((float *)y)[at] = value;
    else
        ((uint16_t *)y)[at] = float_to_bf16_bits(value);
}

int oracle_per_block_dequant(const uint8_t *codes, int64_t ld_codes,
                             const void *scales, int64_t ld_scales,
                             int64_t m_begin, int64_t m_end, int64_t K,
                             int block, int fmt, int mode, int out_fp32,
                             void *y, int64_t ld_y)
{
    if (block != 16 && block != 32 && block != 64 && block != 128)
        return OR_BAD_ARG;
    int rc = check_tile_args(m_end, K, fmt, mode);
    if (rc != OR_OK)
        return rc;
    for (int64_t m = m_begin; m < m_end; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float s = read_scale(scales, ld_scales, mode, OR_LAYOUT_ROW_MAJOR,
                                 m / block, k / block);
            put_output(y, m * ld_y + k, out_fp32,
                       code_value(codes + m * ld_codes, k, fmt) * s);
        }
    return OR_OK;
}

int oracle_per_channel_dequant(const uint8_t *codes, int64_t ld_codes,
                               const void *scales, int64_t m_begin,
                               int64_t m_end, int64_t K, int fmt, int mode,
                               int out_fp32, void *y, int64_t ld_y)
{
    int rc = check_tile_args(m_end, K, fmt, mode);
    if (rc != OR_OK)
        return rc;
    for (int64_t m = m_begin; m < m_end; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float s = read_scale(scales, 0, mode, OR_LAYOUT_ROW_MAJOR, 0, k);
            put_output(y, m * ld_y + k, out_fp32,
                       code_value(codes + m * ld_codes, k, fmt) * s);
        }
    return OR_OK;
}

/* ------------------------------------------- element-level hooks for pins */

/* Saturating RNE encode of n fp32 values (the code step of the cast alone). */
void oracle_encode(const float *q, int64_t n, int fmt, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fmt == OR_FMT_E4M3 ? e4m3_encode(q[i]) : e2m1_encode(q[i]);
}

/* Scale step alone: for each amax, the fp32 scale and the UE8M0 byte
 * (-1 in fp32 mode). */
void oracle_scale(const float *amax, int64_t n, int fmt, int mode,
                  float *s_out, int32_t *ue8m0_out)
{
    for (int64_t i = 0; i < n; ++i) {
        group_scale g = compute_scale(amax[i], fmt, mode);
        s_out[i] = g.s;
        ue8m0_out[i] = g.ue8m0;
    }
}
