/* Exhaustive CPU check of the quantizers' fast scale and reciprocal (test code, not the
 * oracle).
 *
 * For a tile maximum amax in [2^-70, 2^108] the kernels form
 *   s  = RN(amax / 448)  as  q0 = RN(amax * c); e = fma(-q0, 448, amax); s = fma(e, c, q0)
 *        with c = RN(1 / 448) (the correction step of Markstein, IBM J. Res. Develop.
 *        34(1), 1990, with a constant divisor), and
 *   r  = RN(1 / s)       as  y1 = fma(y0, fma(-s, y0, 1), y0); r = fma(y1, fma(-s, y1, 1), y1)
 *        from a hardware approximation y0 of 1 / s (one Newton-Raphson step, then
 *        Markstein's correction step for the reciprocal).
 * The correction step for the reciprocal is known to miss when the significand of s is
 * all ones; the kernels then divide instead, and this program checks that it is the only
 * significand that misses (it skips the reciprocal for it and counts the skips).
 * The hardware approximation is documented to be within one unit in the last place;
 * this program tries every y0 within SPREAD units of the correctly rounded 1 / s, so
 * the check does not depend on which approximation the hardware returns.
 * Both results are compared with the correctly rounded values, decided exactly in
 * binary64 (the products involved have at most 48 significant bits):
 *   s is RN(amax / 448) iff |amax - 448 s| < 224 ulp(s), or = with an even s;
 *   r is RN(1 / s)      iff |1 - s r| < s ulp(r) / 2, or = with an even r.
 * Every positive finite bf16 value in the range is an amax the kernels can meet; the GEMM
 * epilogue also meets binary32 values, for which every significand is checked in
 * [1, 4): inside the range every step above (and its exactness or rounding) scales with
 * powers of two, so one binade of amax covers all, and its scales fill a binade of s.
 * Prints "values_checked mismatches"; exit status 1 on any mismatch.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#define SPREAD 8

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static double ulp(float f) { return (double)nextafterf(f, INFINITY) - (double)f; }

static int is_rn_quotient(float amax, float s) {
    const double d = fabs((double)amax - 448.0 * (double)s);
    const double h = 224.0 * ulp(s);
    return d < h || (d == h && (to_bits(s) & 1u) == 0);
}

static int is_rn_reciprocal(float s, float r) {
    const double d = fabs(1.0 - (double)s * (double)r);
    const double h = (double)s * ulp(r) / 2.0;
    return d < h || (d == h && (to_bits(r) & 1u) == 0);
}

/* Checks one amax; adds to the counters. */
static void check(float amax, unsigned long long *checked, unsigned long long *bad) {
    const float c = 1.0f / 448.0f;
    const float q0 = amax * c;
    const float e = fmaf(-q0, 448.0f, amax);
    const float s = fmaf(e, c, q0);
    ++*checked;
    if (!is_rn_quotient(amax, s) || s != amax / 448.0f) {
        if (*bad < 10) fprintf(stderr, "scale: amax %a s %a want %a\n", amax, s, amax / 448.0f);
        ++*bad;
        return;
    }
    if ((to_bits(s) & 0x7FFFFFu) == 0x7FFFFFu) return;   /* divided by the kernels */
    const float want = 1.0f / s;
    if (!is_rn_reciprocal(s, want)) {
        fprintf(stderr, "reference reciprocal check failed for s %a\n", s);
        ++*bad;
    }
    for (int k = -SPREAD; k <= SPREAD; ++k) {
        const float y0 = from_bits(to_bits(want) + (uint32_t)k);
        const float y1 = fmaf(y0, fmaf(-s, y0, 1.0f), y0);
        const float r = fmaf(y1, fmaf(-s, y1, 1.0f), y1);
        ++*checked;
        if (r != want) {
            if (*bad < 10) fprintf(stderr, "reciprocal: s %a y0 %a got %a want %a\n", s, y0, r, want);
            ++*bad;
        }
    }
}

int main(void) {
    unsigned long long checked = 0, bad = 0;
    for (uint32_t ab = 0x0001; ab < 0x7F80; ++ab) {
        const float amax = from_bits(ab << 16);
        if (!(amax >= 0x1p-70f && amax <= 0x1p+108f)) continue;
        check(amax, &checked, &bad);
    }
#pragma omp parallel for schedule(static) reduction(+ : checked, bad)
    for (uint32_t u = 0x3F800000u; u < 0x40800000u; ++u) {   /* every binary32 in [1, 4) */
        unsigned long long c = 0, b = 0;
        check(from_bits(u), &c, &b);
        checked += c;
        bad += b;
    }
    printf("%llu %llu\n", checked, bad);
    return bad != 0;
}
