/* synth.c -- host implementation of the seeded synthetic inputs (see synth.h). */
#include "synth.h"

#include <math.h>
#include <string.h>

uint64_t tqs_splitmix64(uint64_t seed, uint64_t i)
{
    uint64_t z = seed + (i + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static double uniform01(uint64_t s, uint64_t i)
{
    return ((double)(tqs_splitmix64(s, i) >> 11) + 0.5) * 0x1p-53;
}

double tqs_normal(uint64_t s, uint64_t i)
{
    double u1 = uniform01(s, 2 * i), u2 = uniform01(s, 2 * i + 1);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

double tqs_t5(uint64_t s, uint64_t i)
{
    double z = tqs_normal(s, 6 * i), chi = 0.0;
    for (int k = 1; k <= 5; ++k) {
        double n = tqs_normal(s, 6 * i + k);
        chi += n * n;
    }
    return z / sqrt(chi / 5.0) * sqrt(3.0 / 5.0);
}

static uint16_t to_bf16(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u); /* round to nearest even */
    return (uint16_t)(u >> 16);
}

void tqs_host_kv(uint64_t data_seed, int B, int H, int d, int64_t t_begin, int64_t n, int b_offset,
                 double k_log_sigma, int v_dist, uint16_t *k_out, uint16_t *v_out)
{
    const uint64_t sk = tqs_splitmix64(data_seed, 0), sv = tqs_splitmix64(data_seed, 1);
    const uint64_t ss = tqs_splitmix64(data_seed, 2);
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double cs[512];
            for (int j = 0; j < d; ++j) cs[j] = exp(k_log_sigma * tqs_normal(ss, (uint64_t)h * d + j));
            for (int64_t t = 0; t < n; ++t) {
                const uint64_t base = (((uint64_t)((b + b_offset) * H + h) << 32) + (uint64_t)(t_begin + t)) * (uint64_t)d;
                const int64_t o = (((int64_t)b * H + h) * n + t) * d;
                for (int j = 0; j < d; ++j) {
                    if (k_out) k_out[o + j] = to_bf16(tqs_normal(sk, base + j) * cs[j]);
                    if (v_out)
                        v_out[o + j] = to_bf16(v_dist == TQS_V_T5 ? tqs_t5(sv, base + j) : tqs_normal(sv, base + j));
                }
            }
        }
}

void tqs_host_q(uint64_t data_seed, int64_t step, int B, int QH, int d, uint16_t *q_out)
{
    const uint64_t sq = tqs_splitmix64(data_seed, 3);
    for (int b = 0; b < B; ++b)
        for (int qh = 0; qh < QH; ++qh)
            for (int j = 0; j < d; ++j) {
                const uint64_t e = (((uint64_t)step * B + b) * QH + qh) * (uint64_t)d + j;
                q_out[((int64_t)b * QH + qh) * d + j] = to_bf16(tqs_normal(sq, e));
            }
}
