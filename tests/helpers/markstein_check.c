/* Cross-check of the key kernel's division-free quotient against IEEE division.
 *
 * The kernel computes q = x/scale as q0 = RN(x * RN(1/scale)); e = RN(scale*(-q0) + x)
 * (fused); q = RN(e * RN(1/scale) + q0) (fused) whenever scale is a normal number
 * in [2^-100, 2^100] (Markstein's theorem), and then idx = clip(rint(q - zero)).
 * This program draws bf16 groups of 32 keys over many exponent ranges (including
 * subnormal and near-constant groups), derives scale and zero as the codec does,
 * and counts elements whose index differs from the one IEEE division gives.
 * CPU fmaf and 1.0f/x are IEEE-exact, like the GPU's fused multiply-add and its
 * correctly rounded reciprocal.  Prints "<elements> <mismatches>".
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static uint64_t st = 0x9E3779B97F4A7C15ull;
static uint64_t rnd(void) { st ^= st << 13; st ^= st >> 7; st ^= st << 17; return st; }
static float bf16r(float f)
{
    uint32_t u; memcpy(&u, &f, 4);
    u += 0x7FFF + ((u >> 16) & 1); u &= 0xFFFF0000u;
    float g; memcpy(&g, &u, 4); return g;
}

int main(int argc, char **argv)
{
    long groups = argc > 1 ? atol(argv[1]) : 200000, elems = 0, bad = 0;
    for (long it = 0; it < groups; ++it) {
        float x[32];
        int mode = (int)(it % 4), e0 = (int)(rnd() % 270) - 140;
        for (int j = 0; j < 32; ++j) {
            double v;
            if (mode == 0) v = ldexp((double)((int64_t)(rnd() % 2000001) - 1000000) / 1e6, e0);
            else if (mode == 1) v = ldexp(1.0 + (double)(rnd() % 5) / 128.0, e0) * ((rnd() & 1) ? 1 : -1);
            else if (mode == 2) v = ldexp((double)((int64_t)(rnd() % 2001) - 1000) / 1000.0, e0 + (int)(rnd() % 20));
            else v = ldexp(1.0 + (double)(rnd() % 3) / 128.0, e0);
            x[j] = bf16r((float)v);
            if (isinf(x[j]) || isnan(x[j])) x[j] = 0;
        }
        float mx = x[0], mn = x[0];
        for (int j = 1; j < 32; ++j) { mx = fmaxf(mx, x[j]); mn = fminf(mn, x[j]); }
        for (int signed8 = 0; signed8 < 2; ++signed8) {
            float scale, zero, lo, hi;
            if (signed8) { scale = (mx - mn) / 254.0f; zero = rintf((mx + mn) / (2.0f * scale)); lo = -127; hi = 127; }
            else { scale = (mx - mn) / 15.0f; zero = rintf(mn / scale); lo = 0; hi = 15; }
            if (!(scale >= 0x1p-100f && scale <= 0x1p100f)) continue;
            const float rc = 1.0f / scale;
            for (int j = 0; j < 32; ++j) {
                const float r1 = x[j] / scale - zero;
                const float q0 = x[j] * rc, e = fmaf(-scale, q0, x[j]), q = fmaf(e, rc, q0);
                const float r2 = q - zero;
                ++elems;
                if (rintf(fminf(fmaxf(r1, lo), hi)) != rintf(fminf(fmaxf(r2, lo), hi))) ++bad;
            }
        }
    }
    printf("%ld %ld\n", elems, bad);
    return 0;
}
