// tq_decode.cuh -- fetch kernels: packed cache rows -> bf16 or fp32 K, V.
//
// Method: mlx-bun "TurboQuant -- rotation-based quantization", Part A,
// "Algorithm": keys x_hat = (idx + zero) * scale with the fp16 scale and zero,
// fp32 add before the multiply (the joint K/V decoder paragraph keeps "K's f32
// addition before multiplication"); values x_hat = InvFWHT(centroid[idx] *
// scale) then the sign flip ("apply FWHT then multiply signs", earlier copy of
// the page), the transform normalised by 1/sqrt(d).
//
// GB300 layout.  Keys are elementwise: each thread converts a run of codes
// whose bytes are 4-byte aligned (8 codes at 8/4 bits, 16 at 2 bits, one
// 32-group at 5 bits), so loads and stores of a warp are contiguous.  Values
// need whole rows: one lane owns E = min(d, 128) elements of a row (d/E lanes
// per row), runs the inverse transform in registers (sign and 1/sqrt(d) fused
// into the last multiply) and writes its slice through a padded shared-memory
// slot with a bulk asynchronous store (cp.async.bulk shared -> global).
#pragma once
#include "tq_common.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

// ------------------------------------------------------------------ keys
template <int KB>
struct KeyRun {
    static constexpr int CODES = KB == 8 ? 8 : KB == 4 ? 8 : KB == 2 ? 16 : 32;
    static constexpr int WORDS = CODES * KB / 32;
};

struct KeyDecodeParams {
    const uint8_t *codes;
    const uint16_t *scale, *zero;
    void *out;
    int64_t cap, t0, n, runs;  // runs = B*H*n*d / CODES
    int d;
};

template <int KB, bool F32>
__global__ void __launch_bounds__(256) decode_key_kernel(const __grid_constant__ KeyDecodeParams p)
{
    using R = KeyRun<KB>;
    const int runs_per_row = p.d / R::CODES;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < p.runs; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t orow = i / runs_per_row;  // output row = (bh, t)
        const int ri = (int)(i - orow * runs_per_row);
        const int64_t bh = orow / p.n, t = orow - bh * p.n;
        const int64_t crow = bh * p.cap + p.t0 + t;
        const int e0 = ri * R::CODES;  // first element of the run
        uint32_t w[R::WORDS];
        load_words<R::WORDS, align_of_bytes(R::WORDS * 4)>(p.codes + crow * (p.d * KB / 8) + e0 * KB / 8, w);
        const int g = e0 / 32;
        const float s = f16_bits_to_f32(p.scale[crow * (p.d / 32) + g]);
        const float z = f16_bits_to_f32(p.zero[crow * (p.d / 32) + g]);
        float x[R::CODES];
#pragma unroll
        for (int j = 0; j < R::CODES; ++j) {
            const int bit = j * KB;
            uint32_t c = w[bit >> 5] >> (bit & 31);
            if ((bit & 31) + KB > 32) c |= w[(bit >> 5) + 1] << (32 - (bit & 31));
            c &= (1u << KB) - 1u;
            const float fi = KB == 8 ? (float)(int32_t)(int8_t)c : (float)c;
            x[j] = __fmul_rn(__fadd_rn(fi, z), s);
        }
        const int64_t o = orow * p.d + e0;
        if constexpr (F32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o);
#pragma unroll
            for (int j = 0; j < R::CODES / 4; ++j) dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + o);
#pragma unroll
            for (int j = 0; j < R::CODES / 8; ++j)
                dst[j] = make_uint4(pack_bf16x2(x[8 * j], x[8 * j + 1]), pack_bf16x2(x[8 * j + 2], x[8 * j + 3]),
                                    pack_bf16x2(x[8 * j + 4], x[8 * j + 5]), pack_bf16x2(x[8 * j + 6], x[8 * j + 7]));
        }
    }
}

// ------------------------------------------------------------------ values
constexpr int kVWarps = 4;

template <int D, bool F32>
struct VGeo {
    static constexpr int E = D < 128 ? D : 128;
    static constexpr int LPR = D / E;
    static constexpr int ROWS = 32 / LPR;
    static constexpr int OB = F32 ? 4 : 2;          // output bytes per element
    static constexpr int SLOT = E * OB + 16;        // padded lane slot
    static constexpr int NG = E / 32;
};

struct ValueDecodeParams {
    const uint8_t *codes;
    const uint16_t *scale;
    void *out;
    int H;
    int64_t cap, t0, n, tiles_per_bh, items;
    float inv_sqrt_d;
    float cen[256];
};

template <int E>
__device__ __forceinline__ void fwht_local_d(float (&x)[E])
{
#pragma unroll
    for (int h = 1; h < E; h <<= 1)
#pragma unroll
        for (int i = 0; i < E; i += 2 * h)
#pragma unroll
            for (int j = i; j < i + h; ++j) {
                const float a = x[j], b = x[j + h];
                x[j] = __fadd_rn(a, b);
                x[j + h] = __fsub_rn(a, b);
            }
}

template <int E>
__device__ __forceinline__ void fwht_cross_d(float (&x)[E], int s, bool upper)
{
    const float sg = upper ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, x[j], s);
        x[j] = __fmaf_rn(x[j], sg, other);
    }
}

template <int D, int VB, bool F32>
__global__ void __launch_bounds__(kVWarps * 32) decode_value_kernel(const __grid_constant__ ValueDecodeParams p)
{
    using G = VGeo<D, F32>;
    constexpr int E = G::E;
    extern __shared__ __align__(128) uint8_t smem[];
    float *scen = reinterpret_cast<float *>(smem);
    uint8_t *slots = smem + 1024;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < (1 << VB); i += blockDim.x) scen[i] = p.cen[i];
    __syncthreads();
    const uint32_t slot = smem_addr(slots + (warp * 32 + lane) * G::SLOT);
    const int r = lane / G::LPR, part = lane % G::LPR;

    const int64_t W = (int64_t)gridDim.x * kVWarps;
    for (int64_t item = (int64_t)blockIdx.x * kVWarps + warp; item < p.items; item += W) {
        const int64_t bh = item / p.tiles_per_bh;
        const int64_t t = (item - bh * p.tiles_per_bh) * G::ROWS + r;
        const bool valid = t < p.n;
        const int64_t crow = bh * p.cap + p.t0 + (valid ? t : 0);
        float x[E];
        if (valid) {
            constexpr int LW = E * VB / 32, RB = D * VB / 8, LB = E * VB / 8;
            constexpr int A = align_of_bytes(RB) < align_of_bytes(LB) ? align_of_bytes(RB) : align_of_bytes(LB);
            uint32_t w[LW];
            load_words<LW, A>(p.codes + crow * RB + part * LB, w);
#pragma unroll
            for (int g = 0; g < G::NG; ++g) {
                const float s = f16_bits_to_f32(p.scale[crow * (D / 32) + part * G::NG + g]);
                uint32_t gw[VB], c[32];
#pragma unroll
                for (int k = 0; k < VB; ++k) gw[k] = w[g * VB + k];
                unpack_group<VB>(gw, c);
#pragma unroll
                for (int j = 0; j < 32; ++j) x[32 * g + j] = __fmul_rn(scen[c[j]], s);
            }
        } else {
#pragma unroll
            for (int j = 0; j < E; ++j) x[j] = 0.0f;
        }
        fwht_local_d<E>(x);
        if constexpr (G::LPR >= 2) fwht_cross_d<E>(x, 1, (part & 1) != 0);
        if constexpr (G::LPR >= 4) fwht_cross_d<E>(x, 2, (part & 2) != 0);
        // out = sign * (z * fl(1/sqrt d)); the sign flip is exact, so it is
        // fused into the multiplier
        if constexpr (G::LPR == 1) {
#pragma unroll
            for (int j = 0; j < E; ++j) x[j] = __fmul_rn(x[j], sign_negative(j) ? -p.inv_sqrt_d : p.inv_sqrt_d);
        } else {
#pragma unroll
            for (int wv = 0; wv < E / 32; ++wv) {
                uint32_t m = sign_word(wv);
#pragma unroll
                for (int q = 1; q < G::LPR; ++q)
                    if (part == q) m = sign_word(q * (E / 32) + wv);
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float y = __fmul_rn(x[32 * wv + k], p.inv_sqrt_d);
                    x[32 * wv + k] = __uint_as_float(__float_as_uint(y) ^ ((m << (31 - k)) & 0x80000000u));
                }
            }
        }
        // previous bulk store from this slot must have read it
        bulk_wait_read0();
        if (valid) {
            if constexpr (F32) {
#pragma unroll
                for (int i = 0; i < E / 4; ++i)
                    sts128(slot + 16 * i, make_uint4(__float_as_uint(x[4 * i]), __float_as_uint(x[4 * i + 1]),
                                                     __float_as_uint(x[4 * i + 2]), __float_as_uint(x[4 * i + 3])));
            } else {
#pragma unroll
                for (int i = 0; i < E / 8; ++i)
                    sts128(slot + 16 * i, make_uint4(pack_bf16x2(x[8 * i], x[8 * i + 1]), pack_bf16x2(x[8 * i + 2], x[8 * i + 3]),
                                                     pack_bf16x2(x[8 * i + 4], x[8 * i + 5]),
                                                     pack_bf16x2(x[8 * i + 6], x[8 * i + 7])));
            }
            fence_proxy_async_smem();
            uint8_t *dst = static_cast<uint8_t *>(p.out) + ((bh * p.n + t) * D + part * E) * G::OB;
            bulk_s2g(dst, slot, E * G::OB);
            bulk_commit();
        }
    }
    bulk_wait0();
}

template <int KB, bool F32>
cudaError_t run_key(const CacheView &c, int64_t t0, int64_t n, void *out, cudaStream_t s)
{
    KeyDecodeParams p{};
    p.codes = c.k_codes;
    p.scale = c.k_scale;
    p.zero = c.k_zero;
    p.out = out;
    p.cap = c.cap;
    p.t0 = t0;
    p.n = n;
    p.d = c.d;
    p.runs = (int64_t)c.B * c.H * n * c.d / KeyRun<KB>::CODES;
    const int64_t blocks = (p.runs + 255) / 256;
    const int grid = (int)imin64(blocks, (int64_t)num_sms() * 8);
    decode_key_kernel<KB, F32><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D, int VB, bool F32>
cudaError_t run_value(const CacheView &c, int64_t t0, int64_t n, void *out, cudaStream_t s)
{
    using G = VGeo<D, F32>;
    ValueDecodeParams p{};
    p.codes = c.v_codes;
    p.scale = c.v_scale;
    p.out = out;
    p.H = c.H;
    p.cap = c.cap;
    p.t0 = t0;
    p.n = n;
    p.tiles_per_bh = (n + G::ROWS - 1) / G::ROWS;
    p.items = p.tiles_per_bh * (int64_t)c.B * c.H;
    p.inv_sqrt_d = inv_sqrt_head_dim(D);
    const Tables &tab = codebook_tables(VB);
    for (int i = 0; i < (1 << VB); ++i) p.cen[i] = tab.centroids[i];
    const size_t smem = 1024 + (size_t)kVWarps * 32 * G::SLOT;
    auto kern = decode_value_kernel<D, VB, F32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kVWarps * 32, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t want = (p.items + kVWarps - 1) / kVWarps;
    const int grid = (int)imin64(want, (int64_t)num_sms() * per_sm);
    kern<<<grid, kVWarps * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <bool F32>
cudaError_t key_dispatch(const CacheView &c, int64_t t0, int64_t n, void *out, cudaStream_t s)
{
    switch (c.kb) {
    case 2: return run_key<2, F32>(c, t0, n, out, s);
    case 4: return run_key<4, F32>(c, t0, n, out, s);
    case 5: return run_key<5, F32>(c, t0, n, out, s);
    case 8: return run_key<8, F32>(c, t0, n, out, s);
    }
    return cudaErrorInvalidValue;
}

template <int D, bool F32>
cudaError_t value_dispatch_vb(const CacheView &c, int64_t t0, int64_t n, void *out, cudaStream_t s)
{
    switch (c.vb) {
    case 2: return run_value<D, 2, F32>(c, t0, n, out, s);
    case 3: return run_value<D, 3, F32>(c, t0, n, out, s);
    case 4: return run_value<D, 4, F32>(c, t0, n, out, s);
    case 5: return run_value<D, 5, F32>(c, t0, n, out, s);
    case 8: return run_value<D, 8, F32>(c, t0, n, out, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace tq
