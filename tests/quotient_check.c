/*
 * Exhaustive check of the quotient sequence the CUDA kernel uses for fp32
 * scales:  inv = RN(1/s);  q0 = RN(x*inv);  r = RN(q0*s - x) (fused);
 *          q = RN(q0 - r*inv) (fused)
 * against the IEEE quotient RN(x/s) for every pair the per-token cast can
 * produce: x any finite BF16 value and s = RN(max(a, 1e-4f) / fmt_max) for
 * any finite BF16 amax a >= |x|.
 *   - the two agree bit for bit (signed zeros too), or
 *   - the IEEE quotient is below 2^-64 in magnitude (there the FMA residual
 *     underflows and the correction can miss by an ulp), and then both
 *     quotients carry x's sign and lie below half the format's smallest step
 *     (2^-10 for E4M3, 0.25 for E2M1), so both encode to the same signed
 *     zero -- the code, which is all the cast keeps, is identical.
 * It also evaluates the packed kernels' form of the same sequence, written
 * on negated operands (nx = -x, ninv = -inv):
 *          q0' = RN(nx*ninv);  r' = RN(q0'*s + nx) (fused);
 *          q' = RN(r'*ninv + q0') (fused)
 * and counts the pairs where q' and q differ in any bit (there must be none).
 * Test infrastructure; compiled by tests/test_quotient_proof.py.
 * Usage: quotient_check <fmt_max>
 * Prints "pairs bad tiny tiny_bad form_diff": bad = mismatches with
 * |RN(x/s)| >= 2^-64, tiny = mismatches below it, tiny_bad = those that
 * would change the code, form_diff = pairs where the two forms differ.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float bf16(uint32_t h)
{
    uint32_t u = h << 16;
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
    unsigned long long pairs = 0, bad = 0, sub = 0, sub_bad = 0, form = 0;
    float half_step = fmt_max == 448.0f ? 0x1p-10f : 0.25f;
    for (uint32_t ab = 0; ab <= 0x7F7Fu; ++ab) {
        float a = bf16(ab);
        float ap = a > 1e-4f ? a : 1e-4f;
        float s = ap / fmt_max;
        float inv = 1.0f / s;
        for (uint32_t xb = 0; xb <= ab; ++xb) {
            for (uint32_t sign = 0; sign < 2; ++sign) {
                float x = bf16(xb | (sign << 15));
                float want = x / s;
                float q0 = x * inv;
                /* volatile keeps the compiler from folding the negation of r
                 * into the first FMA, which would not preserve -0 */
                volatile float r = fmaf(q0, s, -x);
                float q = fmaf(-r, inv, q0);
                volatile float nx = -x, ninv = -inv;
                float q0n = nx * ninv;
                float rn = fmaf(q0n, s, nx);
                float qn = fmaf(rn, ninv, q0n);
                if (bits(qn) != bits(q))
                    form++;
                pairs++;
                if (bits(q) == bits(want))
                    continue;
                if (fabsf(want) < 0x1p-64f) {       /* residual underflow */
                    sub++;
                    if (!(fabsf(q) < half_step && fabsf(want) < half_step &&
                          signbit(q) == signbit(x) &&
                          signbit(want) == signbit(x)))
                        sub_bad++;
                    continue;
                }
                if (bad < 5)
                    fprintf(stderr, "x=%a s=%a got %a want %a\n", x, s, q,
                            want);
                bad++;
            }
        }
    }
    printf("%llu %llu %llu %llu %llu\n", pairs, bad, sub, sub_bad, form);
    return 0;
}
