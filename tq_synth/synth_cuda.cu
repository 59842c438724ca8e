// synth_cuda.cu -- device implementation of the seeded synthetic inputs, for
// the multi-gigabyte workloads (definitions in synth.h).  It uses the device's
// own log/cos/sqrt, so a value can differ from the host implementation in the
// last bit of a double; checks against the CPU oracle therefore read the
// generated rows back from the device rather than regenerating them on the host.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

namespace {

__device__ __forceinline__ uint64_t sm64(uint64_t seed, uint64_t i)
{
    uint64_t z = seed + (i + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ double uni(uint64_t s, uint64_t i)
{
    return ((double)(sm64(s, i) >> 11) + 0.5) * 0x1p-53;
}

__device__ __forceinline__ double normal(uint64_t s, uint64_t i)
{
    double u1 = uni(s, 2 * i), u2 = uni(s, 2 * i + 1);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

__device__ __forceinline__ double t5(uint64_t s, uint64_t i)
{
    double z = normal(s, 6 * i), chi = 0.0;
    for (int k = 1; k <= 5; ++k) {
        double n = normal(s, 6 * i + k);
        chi += n * n;
    }
    return z / sqrt(chi / 5.0) * sqrt(3.0 / 5.0);
}

__device__ __forceinline__ uint16_t to_bf16(double x)
{
    float f = (float)x;
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// one thread per (b, h, t, j); output [B][H][n][d] with row stride `ld` elements
__global__ void fill_kv(uint64_t sk, uint64_t sv, uint64_t ss, int B, int H, int d, int64_t t_begin,
                        int64_t n, int b_offset, double k_log_sigma, int v_dist, uint16_t *k_out, uint16_t *v_out)
{
    const int64_t total = (int64_t)B * H * n * d;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(e % d);
        const int64_t t = (e / d) % n;
        const int64_t bh = e / ((int64_t)d * n);
        const int h = (int)(bh % H);
        const uint64_t c = (((uint64_t)(bh + (int64_t)b_offset * H) << 32) + (uint64_t)(t_begin + t)) * (uint64_t)d + j;
        if (k_out) k_out[e] = to_bf16(normal(sk, c) * exp(k_log_sigma * normal(ss, (uint64_t)h * d + j)));
        if (v_out) v_out[e] = to_bf16(v_dist == TQS_V_T5 ? t5(sv, c) : normal(sv, c));
    }
}

__global__ void fill_q(uint64_t sq, int64_t step, int B, int QH, int d, uint16_t *q_out)
{
    const int64_t total = (int64_t)B * QH * d;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x)
        q_out[e] = to_bf16(normal(sq, (uint64_t)step * total + e));
}

uint64_t host_sm64(uint64_t seed, uint64_t i)
{
    uint64_t z = seed + (i + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

}  // namespace

extern "C" int tqs_device_kv(uint64_t data_seed, int B, int H, int d, int64_t t_begin, int64_t n,
                             int b_offset, double k_log_sigma, int v_dist, uint16_t *k_out, uint16_t *v_out,
                             cudaStream_t stream)
{
    fill_kv<<<4096, 256, 0, stream>>>(host_sm64(data_seed, 0), host_sm64(data_seed, 1),
                                      host_sm64(data_seed, 2), B, H, d, t_begin, n, b_offset, k_log_sigma,
                                      v_dist, k_out, v_out);
    return (int)cudaGetLastError();
}

extern "C" int tqs_device_q(uint64_t data_seed, int64_t step, int B, int QH, int d, uint16_t *q_out,
                            cudaStream_t stream)
{
    fill_q<<<256, 256, 0, stream>>>(host_sm64(data_seed, 3), step, B, QH, d, q_out);
    return (int)cudaGetLastError();
}
