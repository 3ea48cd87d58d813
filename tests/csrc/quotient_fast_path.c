/* Exhaustive CPU check of the quantizers' fast quotient (test code, not the oracle).
 *
 * The kernels compute -fl32(x / s) for s = fl32(amax / 448) as
 *     nr = -RN(1 / s); q0n = RN(x * nr); e = fma(q0n, s, x); yn = fma(e, nr, q0n)
 * whenever 2^-80 <= s <= 2^100 (Markstein's correction step on negated operands),
 * round yn to E4M3 and flip the code's sign bit, i.e. they use y = -yn.
 * This program restates that formula with C99 binary32 arithmetic (fmaf rounds once)
 * and compares it with the IEEE quotient x / s over every pair of bf16 values with
 * 0 < amax and |x| <= amax whose scale lies in that range, both signs of x:
 *   - where |x / s| >= 2^-12 the two must be bitwise equal;
 *   - below, both must carry the sign of x and stay below 2^-11, so that both round to
 *     a zero E4M3 code (every magnitude up to 2^-10 does) with that sign. (When x is
 *     about 2^-100 or smaller the residual x - q0 s underflows and the fast quotient may
 *     differ from x / s in its last bits; such quotients are far below the E4M3 range.)
 * A second pass draws random binary32 pairs (the GEMM epilogue quantizes FP32 values):
 * amax with a random significand and an exponent across the fast range of the scale,
 * x = amax times a random binary32 in [-1, 1] (including tiny magnitudes), with the
 * same acceptance rule. The generator is a 64-bit linear congruential sequence per
 * OpenMP chunk, so the pairs do not depend on the thread count.
 * Prints "pairs_checked mismatches"; exit status 1 on any mismatch.
 * Usage: quotient_fast_path [amax_stride [random_pairs_in_millions]]
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static int check_pair(float amax, float x, unsigned long long *bad) {
    const float s = amax / 448.0f;
    const float nr = -(1.0f / s);
    const float q0n = x * nr;
    const float e = fmaf(q0n, s, x);
    const float y = -fmaf(e, nr, q0n);
    const float want = x / s;
    int ok;
    if (fabsf(want) >= 0x1p-12f) ok = to_bits(y) == to_bits(want);
    else ok = signbit(y) == signbit(x) && signbit(want) == signbit(x) && fabsf(y) < 0x1p-11f;
    if (!ok && *bad < 10) fprintf(stderr, "mismatch amax=%a x=%a fast=%a ieee=%a\n", (double)amax, (double)x, (double)y, (double)want);
    return ok;
}

static uint64_t lcg(uint64_t *st) {
    *st = *st * 6364136223846793005ull + 1442695040888963407ull;
    return *st >> 11;
}

int main(int argc, char **argv) {
    const int stride = argc > 1 ? atoi(argv[1]) : 1;
    const long long random_pairs = (argc > 2 ? atoll(argv[2]) : 0) * 1000000ll;
    unsigned long long checked = 0, bad = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(+ : checked, bad)
    for (int ab = 0x0001; ab < 0x7F80; ab += stride) {
        const float amax = from_bits((uint32_t)ab << 16);
        const float s = amax / 448.0f;
        if (!(s >= 0x1p-80f && s <= 0x1p+100f)) continue;
        const float nr = -(1.0f / s);
        for (uint32_t xb = 0; xb <= (uint32_t)ab; ++xb) {
            for (int sign = 0; sign < 2; ++sign) {
                const float x = from_bits((xb << 16) | (sign ? 0x80000000u : 0u));
                const float q0n = x * nr;
                const float e = fmaf(q0n, s, x);
                const float y = -fmaf(e, nr, q0n);
                const float want = x / s;
                ++checked;
                int ok;
                if (fabsf(want) >= 0x1p-12f) ok = to_bits(y) == to_bits(want);
                else ok = signbit(y) == signbit(x) && signbit(want) == signbit(x) && fabsf(y) < 0x1p-11f;
                if (!ok) {
                    if (bad < 10) fprintf(stderr, "mismatch amax=%a x=%a fast=%a ieee=%a\n", (double)amax, (double)x, (double)y, (double)want);
                    ++bad;
                }
            }
        }
    }
    const long long chunks = random_pairs / 65536;
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : checked, bad)
    for (long long c = 0; c < chunks; ++c) {
        uint64_t st = 0x9E3779B97F4A7C15ull ^ (uint64_t)c;
        for (int k = 0; k < 65536; ++k) {
            /* amax: random significand, exponent so that s = amax / 448 lies in [2^-79, 2^99] */
            const uint32_t e_am = 127 - 70 + (uint32_t)(lcg(&st) % 178);
            const float amax = from_bits((e_am << 23) | (uint32_t)(lcg(&st) & 0x7FFFFFu));
            /* x = amax * t, t a random binary32 in [-1, 1] with exponent down to 2^-40 */
            const uint32_t e_t = 127 - (uint32_t)(lcg(&st) % 41);
            float t = from_bits((e_t << 23) | (uint32_t)(lcg(&st) & 0x7FFFFFu));
            if (t > 1.0f) t = 1.0f;
            if (lcg(&st) & 1) t = -t;
            float x = amax * t;
            if (fabsf(x) > amax) x = copysignf(amax, x);
            ++checked;
            if (!check_pair(amax, x, &bad)) ++bad;
        }
    }
    printf("%llu %llu\n", checked, bad);
    return bad != 0;
}
