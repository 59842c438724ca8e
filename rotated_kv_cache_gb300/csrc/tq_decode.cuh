// tq_decode.cuh -- fetch kernels: packed cache rows -> bf16 or fp32 K, V.
//
// Method: mlx-bun "TurboQuant -- rotation-based quantization", Part A,
// "Algorithm": keys x_hat = (idx + zero) * scale with the fp16 scale and zero,
// the fp32 add done before the multiply (the joint K/V decoder paragraph
// keeps that order); values x_hat = InvFWHT(centroid[idx] * scale) followed by
// the sign flip (the page's earlier copy orders the transform before the sign
// multiply), the transform normalised by 1/sqrt(d).
//
// GB300 layout.  Keys are elementwise: a thread converts one 32-group, the
// grid's y axis walks the (sequence, kv-head) pairs, so a warp's loads and
// stores are contiguous and no division is needed.  A code becomes a float
// by placing it in the low mantissa bits of 1.5*2^23 (one byte permute or
// mask); subtracting 1.5*2^23 - zero then gives idx + zero exactly (both are
// integers below 2^24), and the multiply by the scale is the definition's.
// Values need whole rows: as in the encoder a lane holds 64 elements as
// fp32 pairs (element j, element j+32), the row spread over d/64 lanes; the
// inverse transform runs in the definition's stage order with packed .f32x2
// arithmetic, and the sign flip rides on the final multiply by +-1/sqrt(d).
#pragma once
#include "tq_common.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

// ------------------------------------------------------------------ keys
struct KeyDecodeParams {
    const uint8_t *codes;
    const uint16_t *scale, *zero;
    void *out;
    int64_t cap, t0, n, groups_per_bh, BH;
    int d;
};

// 32 codes of one group -> the float bit patterns of 1.5*2^23 + u with u = code
// (unsigned) or code + 128 (signed 8-bit)
template <int KB>
__device__ __forceinline__ void magic_codes(const uint32_t (&w)[KB], uint32_t (&m)[32])
{
    if constexpr (KB == 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t u = w[i] ^ 0x80808080u;  // int8 -> code + 128
#pragma unroll
            for (int k = 0; k < 4; ++k) m[4 * i + k] = __byte_perm(u, 0x4B400000u, 0x7650 + k);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int bit = j * KB, word = bit >> 5, off = bit & 31;
            uint32_t c = (off + KB <= 32) ? (w[word] >> off) : __funnelshift_r(w[word], w[word + 1], off);
            m[j] = (c & ((1u << KB) - 1u)) | 0x4B400000u;
        }
    }
}

// One key group: codes w (KB words), fp16 scale and zero -> 32 outputs at dst
// ((code + zero) * scale in fp32, then bf16 by round to nearest even).
template <int KB, bool F32>
__device__ __forceinline__ void key_group_out(const uint32_t (&w)[KB], float s, float z, void *dst)
{
    // 1.5*2^23 + u - (1.5*2^23 + bias - zero) = idx + zero, exactly
    const float zz = __fsub_rn(KB == 8 ? 12583040.0f : 12582912.0f, z);
    uint32_t m[32];
    magic_codes<KB>(w, m);
    const float2 nz2 = make_float2(-zz, -zz), s2 = make_float2(s, s);
    float2 x[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
        x[k] = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(m[2 * k]), __uint_as_float(m[2 * k + 1])), nz2), s2);
    if constexpr (F32) {
        float *d = static_cast<float *>(dst);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            st_global_v8(d + 8 * j, __float_as_uint(x[4 * j].x), __float_as_uint(x[4 * j].y), __float_as_uint(x[4 * j + 1].x),
                         __float_as_uint(x[4 * j + 1].y), __float_as_uint(x[4 * j + 2].x), __float_as_uint(x[4 * j + 2].y),
                         __float_as_uint(x[4 * j + 3].x), __float_as_uint(x[4 * j + 3].y));
    } else {
        uint16_t *d = static_cast<uint16_t *>(dst);
#pragma unroll
        for (int j = 0; j < 2; ++j)
            st_global_v8(d + 16 * j, pack_bf16x2(x[8 * j].x, x[8 * j].y), pack_bf16x2(x[8 * j + 1].x, x[8 * j + 1].y),
                         pack_bf16x2(x[8 * j + 2].x, x[8 * j + 2].y), pack_bf16x2(x[8 * j + 3].x, x[8 * j + 3].y),
                         pack_bf16x2(x[8 * j + 4].x, x[8 * j + 4].y), pack_bf16x2(x[8 * j + 5].x, x[8 * j + 5].y),
                         pack_bf16x2(x[8 * j + 6].x, x[8 * j + 6].y), pack_bf16x2(x[8 * j + 7].x, x[8 * j + 7].y));
    }
}

template <int KB, bool F32>
__global__ void __launch_bounds__(256) decode_key_kernel(const __grid_constant__ KeyDecodeParams p)
{
    pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    const int64_t gi = (int64_t)blockIdx.x * 256 + threadIdx.x;  // group within the (sequence, kv-head)'s n rows
    if (gi >= p.groups_per_bh) return;
    constexpr int A = align_of_bytes(4 * KB);
    for (int64_t bh = blockIdx.y; bh < p.BH; bh += gridDim.y) {
        // rows t0 .. t0+n-1 of one (sequence, kv-head) are contiguous in every plane
        const int64_t row0 = bh * p.cap + p.t0;
        uint32_t w[KB];
        load_words<KB, A>(p.codes + row0 * (p.d * KB / 8) + gi * (4 * KB), w);
        const int64_t mi = row0 * (p.d / 32) + gi;
        const float s = f16_bits_to_f32(p.scale[mi]), z = f16_bits_to_f32(p.zero[mi]);
        const int64_t o = bh * p.n * p.d + gi * 32;  // whole 32-byte sectors per store
        key_group_out<KB, F32>(w, s, z, static_cast<uint8_t *>(p.out) + o * (F32 ? 4 : 2));
    }
}

// ------------------------------------------------------------------ values
constexpr int kVWarps = 4;

template <int D>
struct VGeo {
    static constexpr int LPR = D / 64;     // lanes per row, 64 elements each
    static constexpr int ROWS = 32 / LPR;  // rows per warp tile
};

struct ValueDecodeParams {
    const uint8_t *codes;
    const uint16_t *scale;
    void *out;
    // keys of the same rows, fetched by the same warps (k_out null: values only)
    const uint8_t *k_codes;
    const uint16_t *k_scale, *k_zero;
    void *k_out;
    int kb;
    int H;
    int64_t cap, t0, n;
    uint32_t tiles_per_bh, items;  // items < 2^31
    FastDiv div_tiles;
    float inv_sqrt_d;
    SignBits sg;  // value signs
    float cen[256];
};

// Byte offset (4 * code) of code j of a group's VB-bit little-endian stream.
template <int VB>
__device__ __forceinline__ uint32_t code_offset(const uint32_t *w, int j)
{
    constexpr uint32_t mask = ((1u << VB) - 1u) << 2;
    const int b = j * VB - 2;  // stream bit that lands on bit 0
    if (b < 0) return (w[0] << -b) & mask;
    const int word = b >> 5, off = b & 31;
    if (off + VB + 2 <= 32) return (w[word] >> off) & mask;
    return __funnelshift_r(w[word], w[word + 1], off) & mask;
}

template <int D, int VB>
__device__ __forceinline__ void load_value_lane(const ValueDecodeParams &p, int64_t crow, int part, uint32_t (&w)[2 * VB],
                                                uint32_t &sc)
{
    constexpr int RB = D * VB / 8, LB = 8 * VB;
    constexpr int A = align_of_bytes(RB) < align_of_bytes(LB) ? align_of_bytes(RB) : align_of_bytes(LB);
    load_words<2 * VB, A>(p.codes + crow * RB + part * LB, w);
    sc = *reinterpret_cast<const uint32_t *>(p.scale + crow * (D / 32) + 2 * part);
}

// The keys of a value tile.  The tile's ROWS rows of one (sequence, kv-head)
// hold 64 key groups, contiguous in every key plane (rows are consecutive);
// lane l fetches groups l and l + 32.  Their loads are issued before the
// tile's value work and consumed after it, so the value work hides them.
struct KeyTile {
    uint32_t w[2][8];
    uint32_t s[2], z[2];  // fp16 bits
};

template <int KB>
__device__ __forceinline__ void key_words_load(const uint8_t *src, uint32_t (&w)[8])
{
    if constexpr (KB == 8) {
        const uint4 a = reinterpret_cast<const uint4 *>(src)[0], b = reinterpret_cast<const uint4 *>(src)[1];
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else if constexpr (KB == 4) {
        const uint4 a = *reinterpret_cast<const uint4 *>(src);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    } else if constexpr (KB == 2) {
        const uint2 a = *reinterpret_cast<const uint2 *>(src);
        w[0] = a.x; w[1] = a.y;
    } else {
#pragma unroll
        for (int i = 0; i < KB; ++i) w[i] = reinterpret_cast<const uint32_t *>(src)[i];
    }
}

template <int D>
__device__ __forceinline__ void key_tile_load(const ValueDecodeParams &p, uint32_t bh, int64_t t_first, int lane,
                                              KeyTile &k)
{
    constexpr int GPR = D / 32;  // groups per row
    const int64_t g0 = ((int64_t)bh * p.cap + p.t0 + t_first) * GPR;  // first group of the tile in the planes
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int g = lane + 32 * i;
        if (t_first + g / GPR >= p.n) continue;
        const int64_t gi = g0 + g;
        switch (p.kb) {
        case 8: key_words_load<8>(p.k_codes + gi * 32, k.w[i]); break;
        case 4: key_words_load<4>(p.k_codes + gi * 16, k.w[i]); break;
        case 5: key_words_load<5>(p.k_codes + gi * 20, k.w[i]); break;
        default: key_words_load<2>(p.k_codes + gi * 8, k.w[i]); break;
        }
        k.s[i] = p.k_scale[gi];
        k.z[i] = p.k_zero[gi];
    }
}

template <int KB, bool F32>
__device__ __forceinline__ void key_group_from_tile(const uint32_t (&w8)[8], uint32_t s, uint32_t z, void *dst)
{
    uint32_t w[KB];
#pragma unroll
    for (int i = 0; i < KB; ++i) w[i] = w8[i];
    key_group_out<KB, F32>(w, f16_bits_to_f32((uint16_t)s), f16_bits_to_f32((uint16_t)z), dst);
}

template <int D, bool F32>
__device__ __forceinline__ void key_tile_store(const ValueDecodeParams &p, uint32_t bh, int64_t t_first, int lane,
                                               const KeyTile &k)
{
    constexpr int GPR = D / 32;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int g = lane + 32 * i;
        if (t_first + g / GPR >= p.n) continue;
        // output [bh][t][D]: group g of the tile starts at element (bh n + t_first) D + 32 g
        void *dst = static_cast<uint8_t *>(p.k_out) + (((int64_t)bh * p.n + t_first) * D + 32 * g) * (F32 ? 4 : 2);
        switch (p.kb) {
        case 8: key_group_from_tile<8, F32>(k.w[i], k.s[i], k.z[i], dst); break;
        case 4: key_group_from_tile<4, F32>(k.w[i], k.s[i], k.z[i], dst); break;
        case 5: key_group_from_tile<5, F32>(k.w[i], k.s[i], k.z[i], dst); break;
        default: key_group_from_tile<2, F32>(k.w[i], k.s[i], k.z[i], dst); break;
        }
    }
}

template <int D, int VB, bool F32>
__global__ void __launch_bounds__(kVWarps * 32, 4) decode_value_kernel(const __grid_constant__ ValueDecodeParams p)
{
    using G = VGeo<D>;
    __shared__ __align__(16) float scen[1 << VB];
    __shared__ __align__(16) float2 smul[G::LPR][34];  // (+-1/sqrt d) of elements (j, j+32) of each part, padded
    pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    for (int i = threadIdx.x; i < (1 << VB); i += blockDim.x) scen[i] = p.cen[i];
    for (int i = threadIdx.x; i < G::LPR * 32; i += blockDim.x) {
        const int part = i >> 5, j = i & 31;
        // elements of P[j] after the transform, and the sign the d128 form leaves on the second
        const int e0 = D == 128 ? 32 * part + j : 64 * part + j, e1 = D == 128 ? 64 + 32 * part + j : e0 + 32;
        const float n1 = D == 128 && part ? -1.0f : 1.0f;
        smul[part][j] = make_float2(sign_negative(p.sg, e0) ? -p.inv_sqrt_d : p.inv_sqrt_d,
                                    n1 * (sign_negative(p.sg, e1) ? -p.inv_sqrt_d : p.inv_sqrt_d));
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane % G::ROWS, part = lane / G::ROWS;
    const char *cen = reinterpret_cast<const char *>(scen);

    const uint32_t W = gridDim.x * kVWarps;
    uint32_t item = blockIdx.x * kVWarps + warp;
    // the next tile's codes are loaded while this one is transformed
    uint32_t nw[2 * VB], nsc = 0;
    auto locate = [&](uint32_t it, int64_t &t, int64_t &crow, uint32_t &bh) {
        bh = fast_div(it, p.div_tiles);
        t = (int64_t)(it - bh * p.tiles_per_bh) * G::ROWS + r;
        crow = (int64_t)bh * p.cap + p.t0 + t;
    };
    if (item < p.items) {
        int64_t t, crow;
        uint32_t bh;
        locate(item, t, crow, bh);
        if (t < p.n) load_value_lane<D, VB>(p, crow, part, nw, nsc);
    }
    for (; item < p.items; item += W) {
        uint32_t w[2 * VB], sc = nsc;
#pragma unroll
        for (int k = 0; k < 2 * VB; ++k) w[k] = nw[k];
        if constexpr (D == 128) {
            if (part) {  // swapped pairs: the second group's codes and scale first
#pragma unroll
                for (int k = 0; k < VB; ++k) {
                    const uint32_t u = w[k];
                    w[k] = w[k + VB];
                    w[k + VB] = u;
                }
                sc = __byte_perm(sc, 0u, 0x1032u);
            }
        }
        int64_t t, crow;
        uint32_t bh;
        locate(item, t, crow, bh);
        const bool valid = t < p.n;
        KeyTile kt;
        const bool keys = p.k_out != nullptr;
        if (keys) key_tile_load<D>(p, bh, t - r, lane, kt);
        if (item + W < p.items) {
            int64_t t1, crow1;
            uint32_t bh1;
            locate(item + W, t1, crow1, bh1);
            if (t1 < p.n) load_value_lane<D, VB>(p, crow1, part, nw, nsc);
        }
        float2 P[32];
        if (valid) {
            const float s0 = f16_bits_to_f32((uint16_t)(sc & 0xFFFFu)), s1 = f16_bits_to_f32((uint16_t)(sc >> 16));
            const float2 s2 = make_float2(s0, s1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float c0 = *reinterpret_cast<const float *>(cen + code_offset<VB>(w, j));
                const float c1 = *reinterpret_cast<const float *>(cen + code_offset<VB>(w + VB, j));
                P[j] = __fmul2_rn(make_float2(c0, c1), s2);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) P[j] = make_float2(0.0f, 0.0f);
        }
        if constexpr (D == 128)
            fwht_pairs_d128<G::ROWS>(P, part);
        else
            fwht_pairs<G::LPR, G::ROWS>(P, part);
        if (valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float4 m = *reinterpret_cast<const float4 *>(&smul[part][j]);
                P[j] = __fmul2_rn(P[j], make_float2(m.x, m.y));
                P[j + 1] = __fmul2_rn(P[j + 1], make_float2(m.z, m.w));
            }
            // P[j].x, P[j].y: elements X0 + j, Y0 + j of the row (whole 32-byte sectors per store)
            constexpr int XS = D == 128 ? 32 : 64, Y0 = D == 128 ? 64 : 32;
            const int64_t o = ((int64_t)bh * p.n + t) * D + XS * part;
            if constexpr (F32) {
                float *dst = static_cast<float *>(p.out) + o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 *q = P + 8 * i;
                    st_global_v8(dst + 8 * i, __float_as_uint(q[0].x), __float_as_uint(q[1].x), __float_as_uint(q[2].x),
                                 __float_as_uint(q[3].x), __float_as_uint(q[4].x), __float_as_uint(q[5].x),
                                 __float_as_uint(q[6].x), __float_as_uint(q[7].x));
                    st_global_v8(dst + Y0 + 8 * i, __float_as_uint(q[0].y), __float_as_uint(q[1].y), __float_as_uint(q[2].y),
                                 __float_as_uint(q[3].y), __float_as_uint(q[4].y), __float_as_uint(q[5].y),
                                 __float_as_uint(q[6].y), __float_as_uint(q[7].y));
                }
            } else {
                uint16_t *dst = static_cast<uint16_t *>(p.out) + o;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float2 *q = P + 16 * i;
                    st_global_v8(dst + 16 * i, pack_bf16x2(q[0].x, q[1].x), pack_bf16x2(q[2].x, q[3].x), pack_bf16x2(q[4].x, q[5].x),
                                 pack_bf16x2(q[6].x, q[7].x), pack_bf16x2(q[8].x, q[9].x), pack_bf16x2(q[10].x, q[11].x),
                                 pack_bf16x2(q[12].x, q[13].x), pack_bf16x2(q[14].x, q[15].x));
                    st_global_v8(dst + Y0 + 16 * i, pack_bf16x2(q[0].y, q[1].y), pack_bf16x2(q[2].y, q[3].y),
                                 pack_bf16x2(q[4].y, q[5].y), pack_bf16x2(q[6].y, q[7].y), pack_bf16x2(q[8].y, q[9].y),
                                 pack_bf16x2(q[10].y, q[11].y), pack_bf16x2(q[12].y, q[13].y), pack_bf16x2(q[14].y, q[15].y));
                }
            }
        }
        if (keys) key_tile_store<D, F32>(p, bh, t - r, lane, kt);
    }
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
    p.groups_per_bh = n * (c.d / 32);
    p.BH = (int64_t)c.B * c.H;
    const int64_t bx = (p.groups_per_bh + 255) / 256;
    if (bx >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)bx, (unsigned)imin64(p.BH, 65535));
    return launch_dependent(decode_key_kernel<KB, F32>, grid, dim3(256), 0, s, p);
}

template <int D, int VB, bool F32>
cudaError_t run_value(const CacheView &c, int64_t t0, int64_t n, void *out, void *k_out, cudaStream_t s)
{
    using G = VGeo<D>;
    ValueDecodeParams p{};
    p.codes = c.v_codes;
    p.scale = c.v_scale;
    p.out = out;
    p.k_codes = c.k_codes;
    p.k_scale = c.k_scale;
    p.k_zero = c.k_zero;
    p.k_out = k_out;
    p.kb = c.kb;
    p.H = c.H;
    p.cap = c.cap;
    p.t0 = t0;
    p.n = n;
    const int64_t tiles = (n + G::ROWS - 1) / G::ROWS, items = tiles * (int64_t)c.B * c.H;
    if (items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    p.tiles_per_bh = (uint32_t)tiles;
    p.items = (uint32_t)items;
    p.div_tiles = make_fastdiv(tiles > 0 ? (uint32_t)tiles : 1u);
    p.inv_sqrt_d = inv_sqrt_head_dim(D);
    p.sg = c.signs;
    const Tables &tab = codebook_tables(VB);
    for (int i = 0; i < (1 << VB); ++i) p.cen[i] = tab.centroids[i];
    auto kern = decode_value_kernel<D, VB, F32>;
    static int per_sm = 0;  // same on every GB300; only a successful query is kept
    if (!per_sm) {
        int k = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, kern, kVWarps * 32, 0);
        if (e != cudaSuccess) return e;
        per_sm = k > 0 ? k : 1;
    }
    const int64_t want = (items + kVWarps - 1) / kVWarps;
    const int grid = (int)imin64(want, (int64_t)num_sms() * per_sm);
    return launch_dependent(kern, dim3((unsigned)grid), dim3(kVWarps * 32), 0, s, p);
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

// Values, and the keys of the same rows when k_out is not null (one launch).
template <int D, bool F32>
cudaError_t value_dispatch_vb(const CacheView &c, int64_t t0, int64_t n, void *out, void *k_out, cudaStream_t s)
{
    switch (c.vb) {
    case 2: return run_value<D, 2, F32>(c, t0, n, out, k_out, s);
    case 3: return run_value<D, 3, F32>(c, t0, n, out, k_out, s);
    case 4: return run_value<D, 4, F32>(c, t0, n, out, k_out, s);
    case 5: return run_value<D, 5, F32>(c, t0, n, out, k_out, s);
    case 8: return run_value<D, 8, F32>(c, t0, n, out, k_out, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace tq
