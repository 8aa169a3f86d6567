/*
 * Exhaustive check of the power-of-two scale exponent the CUDA kernels take
 * from the bits of the floored amax, without dividing:
 *   a' = max(a, 1e-4f) = m * 2^(E-127), m in [1, 2), mantissa field f;
 *   E4M3 (fmt_max 448 = 1.75 * 2^8): e = E - 8 + (f > 0x600000)
 *   E2M1 (fmt_max 6   = 1.5  * 2^2): e = E - 2 + (f > 0x400000)
 * against the definition: r = RN(a' / fmt_max) (IEEE fp32 division), and
 * e = biased exponent of r, plus one when r's mantissa field is nonzero
 * (2^(e-127) is the least power of two >= r).
 * Every positive finite fp32 amax is enumerated (the SwiGLU and RMSNorm
 * casts take the amax of fp32 values, the plain casts of BF16 ones), plus
 * +0.  Test infrastructure; compiled by tests/test_quotient_proof.py.
 * Usage: pow2_exponent_check <fmt_max> [ge]
 * ("ge" tests the wrong rule f >= threshold instead, which must fail.)
 * Prints "values mismatches".
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

int main(int argc, char **argv)
{
    float fmt_max = argc > 1 ? (float)atof(argv[1]) : 448.0f;
    uint32_t drop = fmt_max == 448.0f ? 8u : 2u;
    uint32_t mant_max = fmt_max == 448.0f ? 0x600000u : 0x400000u;
    int ge = argc > 2 && strcmp(argv[2], "ge") == 0;
    unsigned long long values = 0, bad = 0;
    for (uint32_t u = 0;; ++u) {
        float a = from_bits(u);
        float ap = a > 1e-4f ? a : 1e-4f;
        uint32_t r = bits(ap / fmt_max);
        uint32_t want = (r >> 23) + ((r & 0x7FFFFFu) != 0u);
        uint32_t b = bits(ap);
        uint32_t f = b & 0x7FFFFFu;
        uint32_t got = (b >> 23) - drop + (ge ? f >= mant_max : f > mant_max);
        ++values;
        if (got != want) {
            if (bad < 5)
                fprintf(stderr, "amax %a: exponent %u, definition %u\n",
                        (double)a, got, want);
            ++bad;
        }
        if (u == 0x7F7FFFFFu)      /* the largest finite fp32 */
            break;
    }
    printf("%llu %llu\n", values, bad);
    return 0;
}
