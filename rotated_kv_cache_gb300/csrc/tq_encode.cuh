// tq_encode.cuh -- append/encode kernels: bf16 K, V rows -> packed cache rows.
//
// Method: mlx-bun "TurboQuant -- rotation-based quantization", Part A,
// "Algorithm (vllm-metal reference semantics, exact)":
//   keys   per 32-group: signed (8 bits) scale = (max-min)/254, zero =
//          round((max+min)/(2 scale)); unsigned (2/4/5 bits) scale =
//          (max-min)/(2^b-1), zero = round(min/scale); idx = clip(round(x/scale
//          - zero)); fp32 arithmetic, scale/zero stored as fp16.
//   values y = FWHT(x * signs)/sqrt(d); per 32-group rms = sqrt(mean(y^2));
//          idx = searchsorted(boundaries, y/(rms + 1e-8)); little-endian pack.
//
// GB300 layout: one warp processes a tile of token rows of one (sequence,
// kv-head).  Each lane owns E = min(d, 128) consecutive elements of a row
// (d/E lanes per row), brought into a padded shared-memory slot by a bulk
// asynchronous copy (cp.async.bulk, completion on a per-warp mbarrier; two
// slots per warp so the next tile streams in while this one is computed).
// The Walsh-Hadamard transform runs in registers: log2(E) local butterfly
// stages with the sign flip folded in at compile time, then log2(d/E)
// stages across lanes by shuffle.  Stage order and every rounding step follow
// the definition, so codes and scales are reproducible bit for bit.
#pragma once
#include "tq_common.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kWarps = 4;  // warps per CTA

template <int D>
struct Geo {
    static constexpr int E = D < 128 ? D : 128;  // elements per lane
    static constexpr int LPR = D / E;             // lanes per row
    static constexpr int ROWS = 32 / LPR;         // rows per warp tile
    static constexpr int SLOT = E * 2 + 16;       // bytes per lane slot (odd multiple of 16: no bank conflicts)
    static constexpr int TILE = 32 * SLOT;
    static constexpr int NG = E / 32;             // groups per lane
};

struct EncodeParams {
    const uint16_t *src;
    int64_t sb, sh, st;  // element strides of b, h, t
    uint8_t *codes;
    uint16_t *scale, *zero;
    int H;
    int64_t cap, t0, n;
    int64_t tiles_per_bh, items;
    float inv_sqrt_d;
    uint32_t *err;
    float bnd[255];  // value boundaries (ascending)
};

template <int D>
__device__ __forceinline__ void issue_tile(const EncodeParams &p, int64_t item, uint32_t buf, uint32_t bar, int lane)
{
    using G = Geo<D>;
    const int64_t bh = item / p.tiles_per_bh;
    const int64_t t_first = (item - bh * p.tiles_per_bh) * G::ROWS;
    const int rows = (int)imin64(G::ROWS, p.n - t_first);
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(rows * G::LPR * G::E * 2));
    __syncwarp();
    const int r = lane / G::LPR, part = lane % G::LPR;
    if (r < rows) {
        const int64_t b = bh / p.H, h = bh - b * p.H;
        const uint16_t *src = p.src + b * p.sb + h * p.sh + (t_first + r) * p.st + part * G::E;
        bulk_g2s(buf + lane * G::SLOT, src, G::E * 2, bar);
    }
}

// 32 bf16 of a lane slot -> fp32
__device__ __forceinline__ void load_group(uint32_t a, float (&x)[32])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 v = lds128(a + 16 * i);
        x[8 * i + 0] = bf16_lo(v.x); x[8 * i + 1] = bf16_hi(v.x);
        x[8 * i + 2] = bf16_lo(v.y); x[8 * i + 3] = bf16_hi(v.y);
        x[8 * i + 4] = bf16_lo(v.z); x[8 * i + 5] = bf16_hi(v.z);
        x[8 * i + 6] = bf16_lo(v.w); x[8 * i + 7] = bf16_hi(v.w);
    }
}

// ------------------------------------------------------------------ keys
template <int BITS>
__device__ __forceinline__ void key_group(const float (&x)[32], uint32_t (&code)[32], uint16_t &sc, uint16_t &zr)
{
    float mx = x[0], mn = x[0];
#pragma unroll
    for (int j = 1; j < 32; ++j) {
        mx = fmaxf(mx, x[j]);
        mn = fminf(mn, x[j]);
    }
    float scale, zero, lo, hi;
    if constexpr (BITS == 8) {
        scale = __fdiv_rn(__fsub_rn(mx, mn), 254.0f);
        zero = rintf(__fdiv_rn(__fadd_rn(mx, mn), __fmul_rn(2.0f, scale)));
        lo = -127.0f;
        hi = 127.0f;
    } else {
        constexpr float maxv = (float)((1 << BITS) - 1);
        scale = __fdiv_rn(__fsub_rn(mx, mn), maxv);
        zero = rintf(__fdiv_rn(mn, scale));
        lo = 0.0f;
        hi = maxv;
    }
    // idx = clip(round(x/scale - zero)): clip first (NaN -> lo, IEEE maxNum/
    // minNum), then round to nearest even by the 1.5*2^23 shift (|value| <= 127,
    // so the integer lands in the low bits).
    auto code_of = [&](float q) {
        const float c = fminf(fmaxf(__fsub_rn(q, zero), lo), hi);
        const uint32_t t = __float_as_uint(__fadd_rn(c, 12582912.0f)) - 0x4B400000u;
        return BITS == 8 ? (t & 0xFFu) : t;
    };
    if (scale >= 0x1p-100f && scale <= 0x1p100f) {
        // x/scale correctly rounded without a division (Markstein's theorem:
        // with rc = RN(1/scale) and q0 within one ulp of x/scale, q0 + (x -
        // scale*q0)*rc rounds to RN(x/scale)).  Bf16 keys inside a group with
        // max != min keep |x/scale| <= 254*2^8, so nothing overflows; a
        // quotient small enough to be inexact is below 1/4 and rounds to the
        // same code either way.
        const float rc = __frcp_rn(scale);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float q0 = __fmul_rn(x[j], rc);
            const float e = __fmaf_rn(-scale, q0, x[j]);
            code[j] = code_of(__fmaf_rn(e, rc, q0));
        }
    } else {
        // zero, subnormal, huge, Inf or NaN scale: IEEE division
#pragma unroll
        for (int j = 0; j < 32; ++j) code[j] = code_of(__fdiv_rn(x[j], scale));
    }
    sc = f32_to_f16_bits(scale);
    zr = f32_to_f16_bits(zero);
}

template <int D, int BITS>
__device__ __forceinline__ void encode_key_lane(const EncodeParams &p, uint32_t slot, int64_t crow, int part)
{
    using G = Geo<D>;
    constexpr int LW = G::E * BITS / 32;  // output words per lane
    uint32_t w[LW];
    uint16_t sc[G::NG], zr[G::NG];
#pragma unroll
    for (int g = 0; g < G::NG; ++g) {
        float x[32];
        uint32_t code[32];
        load_group(slot + 64 * g, x);
        key_group<BITS>(x, code, sc[g], zr[g]);
        uint32_t gw[BITS];
        pack_group<BITS>(code, gw);
#pragma unroll
        for (int k = 0; k < BITS; ++k) w[g * BITS + k] = gw[k];
    }
    constexpr int RB = D * BITS / 8, LB = G::E * BITS / 8;
    constexpr int A = align_of_bytes(RB) < align_of_bytes(LB) ? align_of_bytes(RB) : align_of_bytes(LB);
    store_words<LW, A>(p.codes + crow * RB + part * LB, w);
    uint32_t sw[G::NG / 2 > 0 ? G::NG / 2 : 1], zw[G::NG / 2 > 0 ? G::NG / 2 : 1];
#pragma unroll
    for (int i = 0; i < G::NG / 2; ++i) {
        sw[i] = (uint32_t)sc[2 * i] | ((uint32_t)sc[2 * i + 1] << 16);
        zw[i] = (uint32_t)zr[2 * i] | ((uint32_t)zr[2 * i + 1] << 16);
    }
    constexpr int SA = align_of_bytes(D / 16) < align_of_bytes(G::NG * 2) ? align_of_bytes(D / 16)
                                                                         : align_of_bytes(G::NG * 2);
    store_words<G::NG / 2, SA>(p.scale + crow * (D / 32) + part * G::NG, sw);
    store_words<G::NG / 2, SA>(p.zero + crow * (D / 32) + part * G::NG, zw);
}

// ------------------------------------------------------------------ values
// Local Sylvester butterflies, strides 1 .. E/2, in place.
template <int E>
__device__ __forceinline__ void fwht_local(float (&x)[E])
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

// Butterflies across lanes: stride E*s pairs lane bit s clear (a) with set (b);
// the clear lane keeps a + b, the set lane a - b.
template <int E>
__device__ __forceinline__ void fwht_cross(float (&x)[E], int lane_bit_s, bool upper)
{
    const float sg = upper ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, x[j], lane_bit_s);
        x[j] = __fmaf_rn(x[j], sg, other);  // exact product: a + b, or a - b
    }
}

template <int NB>
__device__ __forceinline__ uint32_t count_below_linear(const float *bnd, float y)
{
    uint32_t k = 0;
#pragma unroll
    for (int i = 0; i < NB; ++i) k += (bnd[i] < y) ? 1u : 0u;
    return k;
}

// number of boundaries strictly below y (searchsorted, side = left); NaN -> 0
template <int BITS>
__device__ __forceinline__ uint32_t value_index(const EncodeParams &p, const float *sbnd, float y)
{
    if constexpr (BITS <= 3) {
        return count_below_linear<(1 << BITS) - 1>(p.bnd, y);
    } else {
        uint32_t pos = 0;
#pragma unroll
        for (int step = 1 << (BITS - 1); step >= 1; step >>= 1)
            if (sbnd[pos + step - 1] < y) pos += step;
        return pos;
    }
}

template <int D, int BITS>
__device__ __forceinline__ void encode_value_lane(const EncodeParams &p, const float *sbnd, uint32_t slot, int64_t crow,
                                                  int part, bool row_valid)
{
    using G = Geo<D>;
    constexpr int E = G::E;
    float x[E];
    if (row_valid) {
#pragma unroll
        for (int i = 0; i < E / 8; ++i) {
            uint4 v = lds128(slot + 16 * i);
            x[8 * i + 0] = bf16_lo(v.x); x[8 * i + 1] = bf16_hi(v.x);
            x[8 * i + 2] = bf16_lo(v.y); x[8 * i + 3] = bf16_hi(v.y);
            x[8 * i + 4] = bf16_lo(v.z); x[8 * i + 5] = bf16_hi(v.z);
            x[8 * i + 6] = bf16_lo(v.w); x[8 * i + 7] = bf16_hi(v.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < E; ++j) x[j] = 0.0f;
    }
    // x * signs (exact)
    if constexpr (G::LPR == 1) {
#pragma unroll
        for (int j = 0; j < E; ++j) x[j] = x[j] * sign_value(j);
    } else {
#pragma unroll
        for (int w = 0; w < E / 32; ++w) {
            uint32_t m = sign_word(w);
#pragma unroll
            for (int q = 1; q < G::LPR; ++q)
                if (part == q) m = sign_word(q * (E / 32) + w);
#pragma unroll
            for (int k = 0; k < 32; ++k)
                x[32 * w + k] = __uint_as_float(__float_as_uint(x[32 * w + k]) ^ ((m << (31 - k)) & 0x80000000u));
        }
    }
    fwht_local<E>(x);
    if constexpr (G::LPR >= 2) fwht_cross<E>(x, 1, (part & 1) != 0);
    if constexpr (G::LPR >= 4) fwht_cross<E>(x, 2, (part & 2) != 0);
    if (!row_valid) return;

    uint32_t w[E * BITS / 32];
    uint16_t sc[G::NG];
#pragma unroll
    for (int g = 0; g < G::NG; ++g) {
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = __fmul_rn(x[32 * g + j], p.inv_sqrt_d);
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) ss = __fmaf_rn(y[j], y[j], ss);
        const float sigma = __fsqrt_rn(__fdiv_rn(ss, 32.0f));
        const float den = __fadd_rn(sigma, 1e-8f);
        uint32_t code[32];
        if (den < INFINITY) {
            // The index counts the boundaries b below y/den.  Comparing y with
            // b*den instead needs no division; the two can differ only when
            // y/den lies within a few ulps of a boundary.
            if constexpr (BITS <= 3) {
                constexpr int H = 1 << (BITS - 1);  // the table is antisymmetric, b[H-1] = 0
                float P[H - 1];
#pragma unroll
                for (int k = 0; k < H - 1; ++k) P[k] = __fmul_rn(p.bnd[H + k], den);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float a = fabsf(y[j]);
                    uint32_t m = 0;
#pragma unroll
                    for (int k = 0; k < H - 1; ++k) m += a > P[k] ? 1u : 0u;
                    code[j] = y[j] > 0.0f ? H + m : H - 1 - m;
                }
            } else {
                const float rden = __frcp_rn(den);
#pragma unroll
                for (int j = 0; j < 32; ++j) code[j] = value_index<BITS>(p, sbnd, __fmul_rn(y[j], rden));
            }
        } else {
            // non-finite row (Inf/NaN inputs): the definition step by step
#pragma unroll
            for (int j = 0; j < 32; ++j) code[j] = value_index<BITS>(p, sbnd, __fdiv_rn(y[j], den));
        }
        uint32_t gw[BITS];
        pack_group<BITS>(code, gw);
#pragma unroll
        for (int k = 0; k < BITS; ++k) w[g * BITS + k] = gw[k];
        sc[g] = f32_to_f16_bits(sigma);
    }
    constexpr int RB = D * BITS / 8, LB = E * BITS / 8;
    constexpr int A = align_of_bytes(RB) < align_of_bytes(LB) ? align_of_bytes(RB) : align_of_bytes(LB);
    store_words<E * BITS / 32, A>(p.codes + crow * RB + part * LB, w);
    uint32_t sw[G::NG / 2];
#pragma unroll
    for (int i = 0; i < G::NG / 2; ++i) sw[i] = (uint32_t)sc[2 * i] | ((uint32_t)sc[2 * i + 1] << 16);
    constexpr int SA = align_of_bytes(D / 16) < align_of_bytes(G::NG * 2) ? align_of_bytes(D / 16)
                                                                         : align_of_bytes(G::NG * 2);
    store_words<G::NG / 2, SA>(p.scale + crow * (D / 32) + part * G::NG, sw);
}

// ------------------------------------------------------------------ kernel
template <int D, int BITS, bool KEY>
__global__ void __launch_bounds__(kWarps * 32) encode_kernel(const __grid_constant__ EncodeParams p)
{
    using G = Geo<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);  // 2 per warp
    float *sbnd = reinterpret_cast<float *>(smem + 16 * kWarps);
    uint8_t *tiles = smem + 16 * kWarps + (KEY || BITS <= 3 ? 0 : 1024);
    const uint32_t buf0 = smem_addr(tiles + warp * 2 * G::TILE), buf1 = buf0 + G::TILE;
    const uint32_t bar0 = smem_addr(&bars[2 * warp]), bar1 = bar0 + 8;

    if constexpr (!KEY && BITS > 3) {
        for (int i = threadIdx.x; i < (1 << BITS) - 1; i += blockDim.x) sbnd[i] = p.bnd[i];
    }
    if (lane == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar1, 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t W = (int64_t)gridDim.x * kWarps;
    int64_t item = (int64_t)blockIdx.x * kWarps + warp;
    if (item < p.items) issue_tile<D>(p, item, buf0, bar0, lane);
    for (uint32_t k = 0; item < p.items; item += W, ++k) {
        const int64_t next = item + W;
        const uint32_t buf = (k & 1) ? buf1 : buf0, bar = (k & 1) ? bar1 : bar0;
        if (next < p.items) issue_tile<D>(p, next, (k & 1) ? buf0 : buf1, (k & 1) ? bar0 : bar1, lane);
        if (!mbar_wait_bounded(bar, (k >> 1) & 1, p.err)) {
            // give the other copy a bounded chance to land before leaving
            if (next < p.items) mbar_wait_bounded((k & 1) ? bar0 : bar1, ((k + 1) >> 1) & 1, p.err);
            return;
        }
        const int64_t bh = item / p.tiles_per_bh;
        const int64_t t_first = (item - bh * p.tiles_per_bh) * G::ROWS;
        const int r = lane / G::LPR, part = lane % G::LPR;
        const bool valid = t_first + r < p.n;
        const int64_t crow = bh * p.cap + p.t0 + t_first + r;
        const uint32_t slot = buf + lane * G::SLOT;
        if constexpr (KEY) {
            if (valid) encode_key_lane<D, BITS>(p, slot, crow, part);
        } else {
            // every lane of a row joins the cross-lane stages, so no early exit
            encode_value_lane<D, BITS>(p, sbnd, slot, crow, part, valid);
        }
        __syncwarp();
    }
}

template <int D, int BITS, bool KEY>
cudaError_t run(const EncodeParams &p, cudaStream_t s)
{
    using G = Geo<D>;
    const size_t smem = 16 * kWarps + (KEY || BITS <= 3 ? 0 : 1024) + (size_t)kWarps * 2 * G::TILE;
    auto kern = encode_kernel<D, BITS, KEY>;
    static bool configured = false;  // attribute set once per process (idempotent)
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t want = (p.items + kWarps - 1) / kWarps;
    const int grid = (int)imin64(want, (int64_t)num_sms() * per_sm);
    kern<<<grid, kWarps * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_key(int kb, const EncodeParams &p, cudaStream_t s)
{
    switch (kb) {
    case 2: return run<D, 2, true>(p, s);
    case 4: return run<D, 4, true>(p, s);
    case 5: return run<D, 5, true>(p, s);
    case 8: return run<D, 8, true>(p, s);
    }
    return cudaErrorInvalidValue;
}

template <int D>
cudaError_t dispatch_value(int vb, const EncodeParams &p, cudaStream_t s)
{
    switch (vb) {
    case 2: return run<D, 2, false>(p, s);
    case 3: return run<D, 3, false>(p, s);
    case 4: return run<D, 4, false>(p, s);
    case 5: return run<D, 5, false>(p, s);
    case 8: return run<D, 8, false>(p, s);
    }
    return cudaErrorInvalidValue;
}

template <int D>
cudaError_t encode_d(const CacheView &c, const uint16_t *k, const int64_t ks[3], const uint16_t *v,
                     const int64_t vs[3], int64_t t0, int64_t n, cudaStream_t s)
{
    using G = Geo<D>;
    EncodeParams p{};
    p.H = c.H;
    p.cap = c.cap;
    p.t0 = t0;
    p.n = n;
    p.tiles_per_bh = (n + G::ROWS - 1) / G::ROWS;
    p.items = p.tiles_per_bh * (int64_t)c.B * c.H;
    p.inv_sqrt_d = inv_sqrt_head_dim(D);
    p.err = device_error_word();
    if (!p.err) return cudaErrorInvalidDevice;
    const Tables &tab = codebook_tables(c.vb);
    for (int i = 0; i < (1 << c.vb) - 1; ++i) p.bnd[i] = tab.boundaries[i];

    p.src = k;
    p.sb = ks[0]; p.sh = ks[1]; p.st = ks[2];
    p.codes = c.k_codes;
    p.scale = c.k_scale;
    p.zero = c.k_zero;
    cudaError_t e = dispatch_key<D>(c.kb, p, s);
    if (e != cudaSuccess) return e;

    p.src = v;
    p.sb = vs[0]; p.sh = vs[1]; p.st = vs[2];
    p.codes = c.v_codes;
    p.scale = c.v_scale;
    p.zero = nullptr;
    return dispatch_value<D>(c.vb, p, s);
}

}  // namespace
}  // namespace tq
