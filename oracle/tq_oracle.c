/*
 * tq_oracle.c -- plain CPU oracle of the TurboQuant rotated KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA path.
 *
 * Source of every formula: the mlx-bun design page "TurboQuant -- rotation-based
 * quantization", Part A (KV leg), section "Algorithm (vllm-metal reference
 * semantics, exact)", and its earlier copy "turboquant-kv.md", section
 * "Algorithm".  Where the pages leave a step open, the reading taken is stated
 * beside the code.
 *
 * Arithmetic: IEEE binary32, one rounding per operation, in program order
 * (built with -ffp-contract=off and without -ffast-math).  fp16 is used only to
 * store scales and zero points, as the pages fix.  Attention accumulates in
 * binary64.
 *
 * Parity pins (see tests/test_oracle_pins.py): every function below is checked
 * against a value the pages print, a closed form, a textbook table or a library
 * routine.  None is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TQO_OK 0
#define TQO_BAD_ARG 1

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

float tqo_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round-to-nearest-even onto the grid of a binary format with `mant` stored
 * mantissa bits and minimum normal exponent `emin`: the value is scaled to an
 * integer number of grid steps (exact, a power of two), rounded with rint()
 * (ties to even in the default mode), and scaled back. */
static double round_to_grid(double a, int mant, int emin)
{
    int e;
    frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    e -= 1;       /* a in [2^e, 2^(e+1)) */
    if (e < emin) e = emin;
    double step = ldexp(1.0, e - mant);
    return rint(a / step) * step;
}

/* binary32 -> binary16, round to nearest even; NaN -> quiet NaN, overflow -> Inf */
uint16_t tqo_f32_to_f16(float f)
{
    uint16_t s = signbit(f) ? 0x8000u : 0u;
    if (isnan(f)) return (uint16_t)(s | 0x7E00u);
    if (isinf(f)) return (uint16_t)(s | 0x7C00u);
    double a = fabs((double)f);
    if (a == 0.0) return s;
    double r = round_to_grid(a, 10, -14);
    if (r >= 65536.0) return (uint16_t)(s | 0x7C00u);
    if (r == 0.0) return s;
    int e;
    frexp(r, &e);
    e -= 1;
    if (e < -14) /* subnormal: r = k * 2^-24 */
        return (uint16_t)(s | (uint16_t)ldexp(r, 24));
    uint16_t man = (uint16_t)(ldexp(r, -e) * 1024.0 - 1024.0);
    return (uint16_t)(s | (uint16_t)((e + 15) << 10) | man);
}

float tqo_f16_to_f32(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);
    else v = ldexp(1024.0 + m, e - 25);
    return (float)(s ? -v : v);
}

/* binary32 -> bfloat16, round to nearest even (used for the bf16 decode output) */
uint16_t tqo_f32_to_bf16(float f)
{
    uint16_t s = signbit(f) ? 0x8000u : 0u;
    if (isnan(f)) return (uint16_t)(s | 0x7FC0u);
    if (isinf(f)) return (uint16_t)(s | 0x7F80u);
    double a = fabs((double)f);
    if (a == 0.0) return s;
    double r = round_to_grid(a, 7, -126);
    if (r >= 0x1p128) return (uint16_t)(s | 0x7F80u);
    float rf = (float)r; /* exact: r sits on the bf16 grid */
    uint32_t u;
    memcpy(&u, &rf, 4);
    return (uint16_t)(s | (uint16_t)((u >> 16) & 0x7FFFu));
}

/* ------------------------------------------------------------------------ */
/* Sign vector: SplitMix64 (Steele, Lea & Flood, OOPSLA 2014)                */
/* ------------------------------------------------------------------------ */
/* The pages draw the +-1 value signs from a seeded generator and hardcode one
 * vector per head_dim as constants.  The codec here fixes its own generator:
 * output i of SplitMix64 started at `seed`; sign i is -1 when the top bit of
 * that output is set. */
uint64_t tqo_splitmix64(uint64_t seed, uint64_t i)
{
    uint64_t z = seed + (i + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void tqo_sign_vector(int d, uint64_t seed, int8_t *out)
{
    for (int i = 0; i < d; ++i) out[i] = (tqo_splitmix64(seed, (uint64_t)i) >> 63) ? -1 : 1;
}

/* ------------------------------------------------------------------------ */
/* Lloyd-Max codebook for a unit normal                                      */
/* ------------------------------------------------------------------------ */
/* The pages obtain the tables by Lloyd-Max iteration on a unit normal, once,
 * hardcoded; the 3-bit table is printed.  Reading: the optimal quantizer of
 * N(0,1) itself (the fixed point of the two Lloyd-Max conditions), computed on
 * the analytic density rather than on samples:
 *   boundary_i = (c_{i-1} + c_i) / 2                      (nearest neighbour)
 *   c_i        = E[X | boundary_i < X < boundary_{i+1}]   (centroid)
 * Lloyd's iteration alternates the two conditions.  It converges slowly for
 * many levels, so after the Lloyd steps Newton's method is applied to the same
 * two conditions (the fixed point is unique for a log-concave density). */

static double npdf(double x) { return isinf(x) ? 0.0 : exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }
static double ncdf(double x) { return 0.5 * erfc(-x / M_SQRT2); }
static double nsf(double x) { return 0.5 * erfc(x / M_SQRT2); }

/* P(a < X < b), computed on the side of the density where it does not cancel */
static double nprob(double a, double b)
{
    if (a >= 0.0) return nsf(a) - nsf(b);
    if (b <= 0.0) return ncdf(b) - ncdf(a);
    return 1.0 - ncdf(a) - nsf(b);
}

/* E[X | a < X < b] for X ~ N(0,1) */
static double ncentroid(double a, double b) { return (npdf(a) - npdf(b)) / nprob(a, b); }

static void midpoints(int n, const double *c, double *bnd /* n+1 */)
{
    bnd[0] = -INFINITY;
    bnd[n] = INFINITY;
    for (int i = 1; i < n; ++i) bnd[i] = 0.5 * (c[i - 1] + c[i]);
}

/* Lloyd's two steps.  Returns max |change|. */
static double lloyd_step(int n, double *c, double *bnd)
{
    midpoints(n, c, bnd);
    double delta = 0.0;
    for (int i = 0; i < n; ++i) {
        double nc = ncentroid(bnd[i], bnd[i + 1]);
        double dd = fabs(nc - c[i]);
        if (dd > delta) delta = dd;
        c[i] = nc;
    }
    return delta;
}

/* One Newton step on F(c) = T(c) - c, T = centroid-of-midpoint-cells map.
 * dT_i/dc_j is non-zero for j = i-1, i, i+1; with a = lower edge, b = upper
 * edge and g = T_i:  dg/da = pdf(a)(g - a)/P,  dg/db = pdf(b)(b - g)/P, and
 * each edge is the mean of two neighbouring centroids.  Returns max |step|. */
static double newton_step(int n, double *c, double *bnd)
{
    double *lo = malloc(sizeof(double) * n), *di = malloc(sizeof(double) * n);
    double *up = malloc(sizeof(double) * n), *rhs = malloc(sizeof(double) * n);
    midpoints(n, c, bnd);
    for (int i = 0; i < n; ++i) {
        double a = bnd[i], b = bnd[i + 1], P = nprob(a, b);
        double g = (npdf(a) - npdf(b)) / P;
        double ga = isinf(a) ? 0.0 : npdf(a) * (g - a) / P;
        double gb = isinf(b) ? 0.0 : npdf(b) * (b - g) / P;
        lo[i] = 0.5 * ga;              /* d/dc_{i-1} */
        di[i] = 0.5 * ga + 0.5 * gb - 1.0; /* d/dc_i, minus identity */
        up[i] = 0.5 * gb;              /* d/dc_{i+1} */
        rhs[i] = -(g - c[i]);
    }
    /* Thomas algorithm for the tridiagonal system */
    for (int i = 1; i < n; ++i) {
        double w = lo[i] / di[i - 1];
        di[i] -= w * up[i - 1];
        rhs[i] -= w * rhs[i - 1];
    }
    double delta = 0.0;
    double x_next = 0.0;
    for (int i = n - 1; i >= 0; --i) {
        double x = (rhs[i] - (i + 1 < n ? up[i] * x_next : 0.0)) / di[i];
        c[i] += x;
        if (fabs(x) > delta) delta = fabs(x);
        x_next = x;
    }
    free(lo); free(di); free(up); free(rhs);
    return delta;
}

/* Optimal `bits`-bit quantizer of N(0,1): 2^bits centroids (ascending) and
 * 2^bits - 1 boundaries (midpoints), in binary64.  Returns the number of steps
 * taken, or -1 on bad input. */
int tqo_lloyd_max(int bits, double *centroids, double *boundaries)
{
    if (bits < 1 || bits > 8) return -1;
    int n = 1 << bits;
    double *c = centroids, bnd[257];
    for (int i = 0; i < n; ++i) c[i] = -3.0 + 6.0 * (i + 0.5) / n; /* uniform start */
    int steps = 0;
    for (; steps < 400; ++steps)
        if (lloyd_step(n, c, bnd) < 1e-6) break;
    for (int k = 0; k < 60; ++k, ++steps)
        if (newton_step(n, c, bnd) < 1e-15) break;
    /* finish on the Lloyd map itself so the result is its fixed point */
    for (int k = 0; k < 4; ++k, ++steps) lloyd_step(n, c, bnd);
    /* The density is symmetric, so is its optimal quantizer; the pages print
     * the middle 3-bit boundary as exactly 0.  Remove the last-bit asymmetry
     * left by rounding: c_{n-1-i} = -c_i, hence the middle boundary is 0. */
    for (int i = n / 2; i < n; ++i) {
        double m = 0.5 * (c[i] - c[n - 1 - i]);
        c[i] = m;
        c[n - 1 - i] = -m;
    }
    midpoints(n, c, bnd);
    for (int i = 1; i < n; ++i) boundaries[i - 1] = bnd[i];
    return steps;
}

/* fp32 copies used by the codec: centroids rounded, boundaries = midpoint in
 * binary64 of the binary64 centroids, then rounded. */
int tqo_codebook_f32(int bits, float *centroids, float *boundaries)
{
    double c[256], b[255];
    if (tqo_lloyd_max(bits, c, b) < 0) return TQO_BAD_ARG;
    int n = 1 << bits;
    for (int i = 0; i < n; ++i) centroids[i] = (float)c[i];
    for (int i = 0; i < n - 1; ++i) boundaries[i] = (float)b[i];
    return TQO_OK;
}

/* Mean squared error of a quantizer (centroids + boundaries) on N(0,1),
 * integrated in closed form per cell. */
double tqo_normal_mse(int n, const double *c, const double *b)
{
    double mse = 0.0;
    for (int i = 0; i < n; ++i) {
        double lo = i == 0 ? -INFINITY : b[i - 1], hi = i == n - 1 ? INFINITY : b[i];
        double P = nprob(lo, hi);
        double m1 = npdf(lo) - npdf(hi);                       /* E[X; cell]   */
        double m2 = P + (isinf(lo) ? 0.0 : lo * npdf(lo)) - (isinf(hi) ? 0.0 : hi * npdf(hi)); /* E[X^2; cell] */
        mse += m2 - 2.0 * c[i] * m1 + c[i] * c[i] * P;
    }
    return mse;
}

/* ------------------------------------------------------------------------ */
/* Little-endian bitstream (pages: element i occupies bits i*b .. i*b+b-1)   */
/* ------------------------------------------------------------------------ */
/* Reading: bit j of the stream is bit (j mod 8) of byte floor(j/8). */
void tqo_pack_bits(const uint32_t *vals, int n, int bits, uint8_t *out)
{
    memset(out, 0, (size_t)(n * bits + 7) / 8);
    for (int i = 0; i < n; ++i)
        for (int k = 0; k < bits; ++k) {
            int j = i * bits + k;
            if ((vals[i] >> k) & 1u) out[j >> 3] |= (uint8_t)(1u << (j & 7));
        }
}

void tqo_unpack_bits(const uint8_t *in, int n, int bits, uint32_t *vals)
{
    for (int i = 0; i < n; ++i) {
        uint32_t v = 0;
        for (int k = 0; k < bits; ++k) {
            int j = i * bits + k;
            v |= (uint32_t)((in[j >> 3] >> (j & 7)) & 1u) << k;
        }
        vals[i] = v;
    }
}

/* ------------------------------------------------------------------------ */
/* Normalised Walsh-Hadamard transform                                       */
/* ------------------------------------------------------------------------ */
/* Pages: y is the FWHT of x * signs, normalised by 1/sqrt(d); the inverse is
 * the same transform (an involution once normalised).  Reading: Sylvester
 * (natural) order, butterflies (a, b) -> (a + b, a - b) with strides
 * 1, 2, 4, ..., d/2, then every element times fl(1/sqrt(d)). */
void tqo_fwht(float *x, int d)
{
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
    float s = (float)(1.0 / sqrt((double)d));
    for (int j = 0; j < d; ++j) x[j] = x[j] * s;
}

/* ------------------------------------------------------------------------ */
/* Keys: per-32-group asymmetric affine, no rotation                          */
/* ------------------------------------------------------------------------ */
/* clip(): IEEE maxNum/minNum (fmaxf/fminf), so a NaN argument clips to `lo`.
 * The pages leave NaN undefined (its cast is undefined in the reference). */
static int32_t clip_round(float r, float lo, float hi)
{
    float c = fminf(fmaxf(rintf(r), lo), hi);
    return (int32_t)c;
}

/* One group of 32 keys.  bits == 8: signed int8 codes; bits in {2,4,5}:
 * unsigned codes.  Pages:
 *   signed:   max_val = 127; scale = (max - min)/(2 max_val);
 *             zero = round((max + min)/(2 scale)); idx = clip(round(x/scale - zero), -127, 127)
 *   unsigned: max_val = 2^bits - 1; scale = (max - min)/max_val;
 *             zero = round(min/scale); idx = clip(round(x/scale - zero), 0, max_val)
 * all in fp32: the pages compute the affine in fp32 and round only the stored
 * scale and zero to fp16; round = round-half-to-even (rintf).  No
 * epsilon: a constant group gives scale 0 and an infinite (or NaN) zero, the
 * reference defect the pages reproduce on purpose. */
void tqo_key_group(const float *x, int bits, int32_t *idx, uint16_t *scale_h, uint16_t *zero_h)
{
    /* Reading: max/min are IEEE maxNum/minNum folds (a NaN element is
     * skipped; the pages leave NaN inputs open). */
    float mx = x[0], mn = x[0];
    for (int j = 1; j < 32; ++j) {
        mx = fmaxf(mx, x[j]);
        mn = fminf(mn, x[j]);
    }
    float scale, zero, lo, hi;
    if (bits == 8) {
        scale = (mx - mn) / 254.0f;
        zero = rintf((mx + mn) / (2.0f * scale));
        lo = -127.0f;
        hi = 127.0f;
    } else {
        float maxv = (float)((1 << bits) - 1);
        scale = (mx - mn) / maxv;
        zero = rintf(mn / scale);
        lo = 0.0f;
        hi = maxv;
    }
    for (int j = 0; j < 32; ++j) {
        float q = x[j] / scale;
        float r = q - zero;
        idx[j] = clip_round(r, lo, hi);
    }
    *scale_h = tqo_f32_to_f16(scale);
    *zero_h = tqo_f32_to_f16(zero);
}

/* Pages: keys dequantise as (idx + zero) * scale, the fp32 add before the
 * multiply, with the stored fp16 scale and zero. */
void tqo_key_group_dequant(const int32_t *idx, uint16_t scale_h, uint16_t zero_h, float *out)
{
    float s = tqo_f16_to_f32(scale_h), z = tqo_f16_to_f32(zero_h);
    for (int j = 0; j < 32; ++j) out[j] = ((float)idx[j] + z) * s;
}

/* codes of one group -> bytes: int8 two's complement at 8 bits, else the
 * little-endian bitstream of the unsigned codes */
static void key_group_pack(const int32_t *idx, int bits, uint8_t *out)
{
    if (bits == 8) {
        for (int j = 0; j < 32; ++j) out[j] = (uint8_t)(int8_t)idx[j];
    } else {
        uint32_t u[32];
        for (int j = 0; j < 32; ++j) u[j] = (uint32_t)idx[j];
        tqo_pack_bits(u, 32, bits, out);
    }
}

static void key_group_unpack(const uint8_t *in, int bits, int32_t *idx)
{
    if (bits == 8) {
        for (int j = 0; j < 32; ++j) idx[j] = (int8_t)in[j];
    } else {
        uint32_t u[32];
        tqo_unpack_bits(in, 32, bits, u);
        for (int j = 0; j < 32; ++j) idx[j] = (int32_t)u[j];
    }
}

/* ------------------------------------------------------------------------ */
/* Values: sign flip, FWHT, per-32-group RMS, Lloyd-Max index                 */
/* ------------------------------------------------------------------------ */
/* Pages: y = FWHT(x * signs); scale = sqrt(mean(y^2)) per 32-group;
 * y_n = y/(scale + 1e-8); idx = searchsorted(BOUNDARIES, y_n).
 * Readings: the mean is the fp32 sum of squares divided by 32; searchsorted with
 * its default (left) side counts the boundaries strictly below y_n, so a tie
 * goes to the lower cell and NaN gives 0. */
static int32_t searchsorted_left(const float *b, int nb, float y)
{
    int32_t k = 0;
    for (int i = 0; i < nb; ++i)
        if (b[i] < y) ++k;
    return k;
}

/* One row of d values.  y_norm (optional) receives the normalised inputs of
 * the index step, so that tests can find values lying at a boundary. */
void tqo_value_row(const float *x, int d, const int8_t *signs, int bits, const float *boundaries,
                   int32_t *idx, uint16_t *scale_h, float *y_norm)
{
    float y[512];
    for (int j = 0; j < d; ++j) y[j] = x[j] * (float)signs[j];
    tqo_fwht(y, d);
    int nb = (1 << bits) - 1;
    for (int g = 0; g < d / 32; ++g) {
        const float *yg = y + 32 * g;
        /* Reading: the sum of squares is accumulated in element order with a
         * fused multiply-add (one rounding per element). */
        float ss = 0.0f;
        for (int j = 0; j < 32; ++j) ss = fmaf(yg[j], yg[j], ss);
        float sigma = sqrtf(ss / 32.0f);
        float den = sigma + 1e-8f;
        for (int j = 0; j < 32; ++j) {
            float yn = yg[j] / den;
            if (y_norm) y_norm[32 * g + j] = yn;
            idx[32 * g + j] = searchsorted_left(boundaries, nb, yn);
        }
        scale_h[g] = tqo_f32_to_f16(sigma);
    }
}

/* Pages: x_hat = InvFWHT(centroids[idx] * scale * signs^-1), i.e. "apply FWHT
 * then multiply signs" (the earlier copy of the page spells out the order).
 * Reading: the stored fp16 scale, upcast, without the 1e-8. */
void tqo_value_row_dequant(const int32_t *idx, const uint16_t *scale_h, int d, const int8_t *signs,
                           const float *centroids, float *out)
{
    float y[512];
    for (int j = 0; j < d; ++j) y[j] = centroids[idx[j]] * tqo_f16_to_f32(scale_h[j / 32]);
    tqo_fwht(y, d);
    for (int j = 0; j < d; ++j) out[j] = y[j] * (float)signs[j];
}

/* Deferred fetch (page section "Deferred inverse FWHT": attention is linear in
 * V, so the weighted sum can be formed in the rotated domain and brought back
 * once per output row): the value row before the inverse transform,
 * centroid[idx] * rms -- the first step of tqo_value_row_dequant. */
void tqo_value_row_rotated(const int32_t *idx, const uint16_t *scale_h, int d, const float *centroids, float *out)
{
    for (int j = 0; j < d; ++j) out[j] = centroids[idx[j]] * tqo_f16_to_f32(scale_h[j / 32]);
}

/* The page's unrotateValues: a vector formed in the rotated domain back to
 * the model's basis, signs * FWHT(x)/sqrt(d) -- the second half of
 * tqo_value_row_dequant, in the same order. */
void tqo_unrotate(const float *x, int d, const int8_t *signs, float *out)
{
    float y[512];
    for (int j = 0; j < d; ++j) y[j] = x[j];
    tqo_fwht(y, d);
    for (int j = 0; j < d; ++j) out[j] = y[j] * (float)signs[j];
}

/* ------------------------------------------------------------------------ */
/* Whole-cache operations on the plane layout                                 */
/* ------------------------------------------------------------------------ */
/* Planes, all [B][H][cap][...] row-major:
 *   k_codes [d*kb/8] bytes, k_scale [d/32] fp16, k_zero [d/32] fp16,
 *   v_codes [d*vb/8] bytes, v_scale [d/32] fp16.
 * Pages: groups run along head_dim only, so token slices stay byte-safe. */
static int valid_dims(int d, int kb, int vb)
{
    if (!(d == 64 || d == 128 || d == 256 || d == 512)) return 0;
    if (!(kb == 2 || kb == 4 || kb == 5 || kb == 8)) return 0;
    if (!(vb == 2 || vb == 3 || vb == 4 || vb == 5 || vb == 8)) return 0;
    return 1;
}

/* Bytes per token per kv-head: K codes + K scale/zero + V codes + V scale. */
int64_t tqo_bytes_per_token_head(int d, int kb, int vb)
{
    return (int64_t)d * kb / 8 + 2 * 2 * (d / 32) + (int64_t)d * vb / 8 + 2 * (d / 32);
}

/* Encode n tokens of K and V (bf16, [B][H][n][d] contiguous) into rows
 * [t0, t0+n) of the planes. */
int tqo_encode(int B, int H, int d, int kb, int vb, int64_t cap, int64_t t0, int64_t n,
               const uint16_t *k, const uint16_t *v, const int8_t *signs, const float *boundaries,
               uint8_t *k_codes, uint16_t *k_scale, uint16_t *k_zero, uint8_t *v_codes, uint16_t *v_scale)
{
    if (!valid_dims(d, kb, vb) || t0 < 0 || n < 0 || t0 + n > cap) return TQO_BAD_ARG;
    const int g = d / 32;
    const int64_t kr = (int64_t)d * kb / 8, vr = (int64_t)d * vb / 8;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int64_t t = 0; t < n; ++t) {
                const int64_t src = (((int64_t)b * H + h) * n + t) * d;
                const int64_t row = ((int64_t)b * H + h) * cap + t0 + t;
                float x[512];
                int32_t idx[512];
                for (int j = 0; j < d; ++j) x[j] = tqo_bf16_to_f32(k[src + j]);
                for (int gi = 0; gi < g; ++gi) {
                    tqo_key_group(x + 32 * gi, kb, idx, &k_scale[row * g + gi], &k_zero[row * g + gi]);
                    key_group_pack(idx, kb, k_codes + row * kr + gi * 4 * kb);
                }
                for (int j = 0; j < d; ++j) x[j] = tqo_bf16_to_f32(v[src + j]);
                tqo_value_row(x, d, signs, vb, boundaries, idx, &v_scale[row * g], NULL);
                uint32_t u[512];
                for (int j = 0; j < d; ++j) u[j] = (uint32_t)idx[j];
                tqo_pack_bits(u, d, vb, v_codes + row * vr);
            }
    return TQO_OK;
}

/* Decode rows [t0, t0+n) to fp32 [B][H][n][d] (either output may be NULL). */
int tqo_decode(int B, int H, int d, int kb, int vb, int64_t cap, int64_t t0, int64_t n,
               const uint8_t *k_codes, const uint16_t *k_scale, const uint16_t *k_zero,
               const uint8_t *v_codes, const uint16_t *v_scale, const int8_t *signs,
               const float *centroids, float *k_out, float *v_out)
{
    if (!valid_dims(d, kb, vb) || t0 < 0 || n < 0 || t0 + n > cap) return TQO_BAD_ARG;
    const int g = d / 32;
    const int64_t kr = (int64_t)d * kb / 8, vr = (int64_t)d * vb / 8;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int64_t t = 0; t < n; ++t) {
                const int64_t dst = (((int64_t)b * H + h) * n + t) * d;
                const int64_t row = ((int64_t)b * H + h) * cap + t0 + t;
                int32_t idx[512];
                if (k_out)
                    for (int gi = 0; gi < g; ++gi) {
                        key_group_unpack(k_codes + row * kr + gi * 4 * kb, kb, idx);
                        tqo_key_group_dequant(idx, k_scale[row * g + gi], k_zero[row * g + gi],
                                              k_out + dst + 32 * gi);
                    }
                if (v_out) {
                    uint32_t u[512];
                    tqo_unpack_bits(v_codes + row * vr, d, vb, u);
                    for (int j = 0; j < d; ++j) idx[j] = (int32_t)u[j];
                    tqo_value_row_dequant(idx, &v_scale[row * g], d, signs, centroids, v_out + dst);
                }
            }
    return TQO_OK;
}

/* Rows [t0, t0+n) of the value planes in the rotated domain (fp32). */
int tqo_decode_rotated(int B, int H, int d, int vb, int64_t cap, int64_t t0, int64_t n, const uint8_t *v_codes,
                       const uint16_t *v_scale, const float *centroids, float *v_out)
{
    if (!valid_dims(d, 8, vb) || t0 < 0 || n < 0 || t0 + n > cap) return TQO_BAD_ARG;
    const int g = d / 32;
    const int64_t vr = (int64_t)d * vb / 8;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int64_t t = 0; t < n; ++t) {
                const int64_t dst = (((int64_t)b * H + h) * n + t) * d;
                const int64_t row = ((int64_t)b * H + h) * cap + t0 + t;
                int32_t idx[512];
                uint32_t u[512];
                tqo_unpack_bits(v_codes + row * vr, d, vb, u);
                for (int j = 0; j < d; ++j) idx[j] = (int32_t)u[j];
                tqo_value_row_rotated(idx, &v_scale[row * g], d, centroids, v_out + dst);
            }
    return TQO_OK;
}

/* Decode attention over the dequantised cache, the plain definition:
 *   S_t = (sum_j q_j k_hat_{t,j}) * softmax_scale,  p = softmax(S),  o = sum_t p_t v_hat_t
 * for t in [0, seq_len), with q-head h reading kv-head h / (QH/H) (GQA by
 * whole-head replication).  k_hat and v_hat are the fp32 dequantised rows
 * (eager: values un-rotated before the sum); the sums run in binary64.
 * Only the (b, q-head) pairs with want[b*QH + qh] != 0 are computed (want may
 * be NULL for all). */
int tqo_attention(int B, int H, int d, int kb, int vb, int64_t cap,
                  const uint8_t *k_codes, const uint16_t *k_scale, const uint16_t *k_zero,
                  const uint8_t *v_codes, const uint16_t *v_scale, const int8_t *signs,
                  const float *centroids, const uint16_t *q, int QH, int64_t seq_len,
                  double softmax_scale, const uint8_t *want, double *out)
{
    if (!valid_dims(d, kb, vb) || QH <= 0 || QH % H != 0 || seq_len < 1 || seq_len > cap)
        return TQO_BAD_ARG;
    const int G = QH / H, g = d / 32;
    const int64_t kr = (int64_t)d * kb / 8, vr = (int64_t)d * vb / 8;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int qh = 0; qh < QH; ++qh) {
            if (want && !want[b * QH + qh]) continue;
            const int h = qh / G;
            double qv[512], acc[512], *s = malloc(sizeof(double) * (size_t)seq_len);
            float kh[512], vh[512];
            int32_t idx[512];
            uint32_t u[512];
            for (int j = 0; j < d; ++j) qv[j] = tqo_bf16_to_f32(q[((int64_t)b * QH + qh) * d + j]);
            double m = -INFINITY;
            for (int64_t t = 0; t < seq_len; ++t) {
                const int64_t row = ((int64_t)b * H + h) * cap + t;
                for (int gi = 0; gi < g; ++gi) {
                    key_group_unpack(k_codes + row * kr + gi * 4 * kb, kb, idx);
                    tqo_key_group_dequant(idx, k_scale[row * g + gi], k_zero[row * g + gi], kh + 32 * gi);
                }
                double dot = 0.0;
                for (int j = 0; j < d; ++j) dot += qv[j] * (double)kh[j];
                s[t] = dot * softmax_scale;
                if (s[t] > m) m = s[t];
            }
            double l = 0.0;
            for (int j = 0; j < d; ++j) acc[j] = 0.0;
            for (int64_t t = 0; t < seq_len; ++t) {
                const int64_t row = ((int64_t)b * H + h) * cap + t;
                double p = exp(s[t] - m);
                l += p;
                tqo_unpack_bits(v_codes + row * vr, d, vb, u);
                for (int j = 0; j < d; ++j) idx[j] = (int32_t)u[j];
                tqo_value_row_dequant(idx, &v_scale[row * g], d, signs, centroids, vh);
                for (int j = 0; j < d; ++j) acc[j] += p * (double)vh[j];
            }
            for (int j = 0; j < d; ++j) out[((int64_t)b * QH + qh) * d + j] = acc[j] / l;
            free(s);
        }
    return TQO_OK;
}
