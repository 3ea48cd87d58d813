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
 * Prints "pairs_checked mismatches"; exit status 1 on any mismatch.
 * Usage: quotient_fast_path [amax_stride]
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

int main(int argc, char **argv) {
    const int stride = argc > 1 ? atoi(argv[1]) : 1;
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
    printf("%llu %llu\n", checked, bad);
    return bad != 0;
}
