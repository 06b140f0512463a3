/*
 * Check of the fp8 cache's quotient method (test helper, plain C).
 *
 * The fp8 cache stores e4m3(RN32(x / s)).  The GPU computes the quotient without a
 * division per value: with y = RN(1/s), q0 = RN(|x| y) and two Markstein correction
 * steps q' = RN(q + RN(|x| - q s) y) (fused multiply-adds; Markstein, "Computation of
 * elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
 * 1990), for scales in [2^-64, 2^64].  This program restates that method with C's fmaf
 * and compares the resulting e4m3 codes with those of the IEEE quotient |x| / s, over
 * every positive finite bf16 x and random fp32 x, for a list of scales.
 *
 * The kernels evaluate the same steps on the signed value with the negated reciprocal
 * -y: p0 = RN(x (-y)), p' = RN(p + RN(x + p s) (-y)).  Each p is the exact negation of
 * the step above for x (nearest-even rounding is symmetric), so the codes of x / s are
 * those of p2 with the sign bit flipped; zeros come out with the opposite sign of x,
 * which the flip turns into the sign of x.  A NaN code (a non-finite x, or a product
 * that overflows) sends the value to the unsigned form with the sign carried.  The
 * second check compares that form's signed codes with those of the IEEE quotient x / s
 * over every finite and infinite bf16 x of both signs and random fp32 x of both signs.
 * It prints the number of pairs and of code mismatches, summed over both checks.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float f_of(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }

static uint64_t state = 88172645463325252ull;
static uint64_t next(void) { state ^= state << 13; state ^= state >> 7; state ^= state << 17; return state; }

/* e4m3 code of a non-negative float: nearest even on the e4m3 grid, saturating at 448 */
static int e4m3_code(float v)
{
    double a = v, r, f;
    int k, e, E;
    if (isnan(v)) return 0x7F;
    if (a >= 448.0) return 0x7E;
    if (a == 0.0) return 0;
    frexp(a, &k);
    k -= 1;
    if (k < -6) k = -6;
    r = nearbyint(a / ldexp(1.0, k - 3)) * ldexp(1.0, k - 3);
    if (r >= 448.0) return 0x7E;
    if (r == 0.0) return 0;
    f = frexp(r, &e);
    E = e - 1 + 7;
    if (E <= 0) return (int)(r / ldexp(1.0, -9));
    return (E << 3) | (int)((f * 2.0 - 1.0) * 8.0 + 0.5);
}

static float method(float a, float s, float y)
{
    float q0 = a * y, q1, q2;
    if (!(q0 <= 3.40282347e38f)) return q0;
    q1 = fmaf(fmaf(-q0, s, a), y, q0);
    q2 = fmaf(fmaf(-q1, s, a), y, q1);
    return q2;
}

/* e4m3 code of any float, sign kept (NaN: sign | 0x7F) */
static int e4m3_signed(float v)
{
    return (signbit(v) ? 0x80 : 0) | e4m3_code(fabsf(v));
}

/* The signed form with the negated reciprocal ny = -y, and its fallback. */
static int method_signed_code(float x, float s, float y)
{
    float ny = -y;
    float p0 = x * ny;
    float p1 = fmaf(fmaf(p0, s, x), ny, p0);
    float p2 = fmaf(fmaf(p1, s, x), ny, p1);
    int code = e4m3_signed(p2) ^ 0x80;
    if ((code & 0x7F) == 0x7F)
        code = e4m3_signed(copysignf(method(fabsf(x), s, y), x));
    return code;
}

static long long check_signed(float x, float s, float y)
{
    return e4m3_signed(x / s) != method_signed_code(x, s, y);
}

int main(int argc, char **argv)
{
    int nscales = argc > 1 ? atoi(argv[1]) : 200, nrand = argc > 2 ? atoi(argv[2]) : 20000;
    static const float fixed[] = {0x1p-64f, 0x1p64f, 3.0f, 1.0f / 3.0f, 0.37f, 0.01f, 1.0f,
                                  1.99999988f, 1.00000012f, 0.0078125f, 448.0f};
    int nfixed = (int)(sizeof(fixed) / sizeof(fixed[0]));
    long long pairs = 0, bad = 0;
    int k, i;
    uint32_t h;
    for (k = 0; k < nfixed + nscales; k++) {
        float s = k < nfixed ? fixed[k]
                             : f_of(((uint32_t)((int)(next() % 129) - 64 + 127) << 23) |
                                    (uint32_t)(next() & 0x7FFFFF));
        float y = 1.0f / s;
        for (h = 0; h < 0x7F80; h++) {          /* every positive finite bf16 */
            float a = f_of(h << 16);
            pairs++;
            if (e4m3_code(a / s) != e4m3_code(method(a, s, y))) bad++;
        }
        for (i = 0; i < nrand; i++) {            /* random positive finite fp32 */
            float a = f_of((uint32_t)(next() % 0x7F800000u));
            pairs++;
            if (e4m3_code(a / s) != e4m3_code(method(a, s, y))) bad++;
        }
        for (h = 0; h < 0x10000; h++) {         /* every bf16 but NaN, both signs */
            float x = f_of(h << 16);
            if (isnan(x)) continue;
            pairs++;
            bad += check_signed(x, s, y);
        }
        for (i = 0; i < nrand; i++) {            /* random finite fp32, both signs */
            float x = f_of((uint32_t)(next() % 0x7F800000u) | (uint32_t)(next() & 1) << 31);
            pairs++;
            bad += check_signed(x, s, y);
        }
    }
    printf("%lld %lld\n", pairs, bad);
    return 0;
}
