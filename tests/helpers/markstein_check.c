/* Cross-check of the key kernel's division-free quotient against IEEE division.
 *
 * The kernel computes q = x/scale as q0 = RN(x * RN(1/scale)); e = RN(scale*(-q0) + x)
 * (fused); q = RN(e * RN(1/scale) + q0) (fused) whenever scale is a normal number
 * in [2^-100, 2^100] (Markstein's theorem), and then idx = clip(rint(q - zero)).
 * This program draws bf16 groups of 32 keys over many exponent ranges (including
 * subnormal and near-constant groups), derives scale and zero as the codec does,
 * and counts elements whose index differs from the one IEEE division gives.
 * CPU fmaf and 1.0f/x are IEEE-exact, like the GPU's fused multiply-add and its
 * correctly rounded reciprocal.
 *
 * The per-group parameters are checked the same way, bit for bit (the sign of
 * a zero included): scale = (max-min)/C for C in {254, 3, 15, 31} through the
 * constant reciprocal RN(1/C) whenever max-min lies in [2^-100, 2^100], the
 * signed zero point (max+min)/(2 scale) through RN(1/scale)/2, and the unsigned
 * zero point min/scale through RN(1/scale).  Prints "<elements> <mismatches>
 * <groups> <parameter mismatches>".
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

static uint32_t bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static float markstein(float x, float y, float ry)
{
    const float q0 = x * ry, e = fmaf(-y, q0, x);
    return fmaf(e, ry, q0);
}

/* 1 if any per-group parameter from the division-free forms differs from IEEE division */
static int params_differ(float mx, float mn)
{
    static const float C[4] = {254.0f, 3.0f, 15.0f, 31.0f};
    const float d = mx - mn;
    if (!(d >= 0x1p-100f && d <= 0x1p100f)) return 0;
    int bad = 0;
    for (int c = 0; c < 4; ++c) {
        const float scale = d / C[c];
        bad |= bits(markstein(d, C[c], 1.0f / C[c])) != bits(scale);
        if (!(scale >= 0x1p-100f && scale <= 0x1p100f)) continue;
        const float rc = 1.0f / scale;
        if (c == 0) bad |= bits(rintf(markstein(mx + mn, 2.0f * scale, 0.5f * rc))) != bits(rintf((mx + mn) / (2.0f * scale)));
        else bad |= bits(rintf(markstein(mn, scale, rc))) != bits(rintf(mn / scale));
    }
    return bad;
}

int main(int argc, char **argv)
{
    long groups = argc > 1 ? atol(argv[1]) : 200000, elems = 0, bad = 0, pgroups = 0, pbad = 0;
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
        ++pgroups;
        pbad += params_differ(mx, mn);
        {   /* arbitrary fp32 max/min pairs as well (not only bf16 groups) */
            uint32_t a = (uint32_t)rnd(), b = (uint32_t)rnd();
            float fa, fb; memcpy(&fa, &a, 4); memcpy(&fb, &b, 4);
            if (isfinite(fa) && isfinite(fb)) { ++pgroups; pbad += params_differ(fmaxf(fa, fb), fminf(fa, fb)); }
        }
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
    printf("%ld %ld %ld %ld\n", elems, bad, pgroups, pbad);
    return 0;
}
