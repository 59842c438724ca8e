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
// GB300 layout.  A warp processes a tile of token rows of one (sequence,
// kv-head); each row reaches shared memory by one bulk asynchronous copy
// (cp.async.bulk, completion on a per-warp mbarrier, two tiles in flight per
// warp).  A row is split over LPR lanes, lane = part * ROWS + row:
//   keys    32 elements per lane = one quantisation group, so the group's
//           max/min, scale and zero point never leave the lane;
//   values  64 elements per lane = two RMS groups, held as fp32 pairs
//           (element j, element j+32).  Butterfly strides 1..16 run on the
//           pairs with packed .f32x2 arithmetic, stride 32 inside each pair,
//           strides 64.. across the row's lanes by shuffle; the two groups'
//           sums of squares run as one packed chain.
// Every rounding step is the definition's, in its order: codes, scales and
// zero points are reproducible bit for bit, except a value index whose
// normalised input lies within a few ulps of a boundary (thresholds are
// compared instead of dividing).
#pragma once
#include "tq_common.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kWarps = 4;  // warps per CTA
constexpr int kKeyRows = 2;  // key rows (groups) per lane in a warp tile: independent chains that interleave

template <int D, bool KEY, int KR = kKeyRows>
struct EGeo {
    static constexpr int E = KEY ? 32 : 64;   // elements per lane and row
    static constexpr int LPR = D / E;          // lanes per row
    static constexpr int ROWS = 32 / LPR;      // rows one pass of the warp covers
    static constexpr int RPL = KEY ? KR : 1;   // rows per lane: independent key groups interleave
    static constexpr int TROWS = ROWS * RPL;   // rows per warp tile
    // Two tile layouts, one read formula (chunk k of a row's 64-column box at
    // base + 16 * (k ^ xr)):
    //   tensor copy  D/64 boxes of TROWS x 128 bytes, 128-byte swizzle (xr = row & 7)
    //   row copies   rows RS bytes apart, RS = 16 mod 128 (xr = 0)
    // either way 8 rows' 16-byte reads hit 8 different bank groups.
    static constexpr int RS = 2 * D + 16;
    static constexpr int BOX = (TROWS * 128 + 1023) / 1024 * 1024;  // box stride: swizzle atoms are 1024-aligned
    static constexpr int TILE = ((TROWS * RS > (D / 64) * BOX ? TROWS * RS : (D / 64) * BOX) + 1023) / 1024 * 1024;
    static constexpr int MTAB = KEY ? 0 : LPR * 272;  // value sign masks: 16 x 16 bytes (+16 pad) per part
};

// value tiles stage their packed codes (ROWS rows x row bytes, 16-byte multiple)
template <int D, int BITS>
struct VStage {
    static constexpr int RB = D * BITS / 8;
    static constexpr int BYTES = (EGeo<D, false>::ROWS * RB + 15) / 16 * 16;
};

struct EncodeParams {
    const uint16_t *src;
    int64_t sb, sh, st;  // element strides of b, h, t
    uint8_t *codes;
    uint16_t *scale, *zero;
    int H;
    int64_t cap, t0, n;
    uint32_t tiles_per_bh, items;  // items < 2^31
    FastDiv div_tiles, div_h;      // x / tiles_per_bh, x / H
    float inv_sqrt_d;
    SignBits sg;  // value signs
    uint32_t *err;
    int use_tma;     // tiles arrive by tensor copies of the map (else one bulk copy per row)
    float bnd[255];  // value boundaries (ascending)
};

// Bytes a tile's copies bring into shared memory.
template <int D, bool KEY, int KR = kKeyRows>
__device__ __forceinline__ uint32_t tile_bytes(const EncodeParams &p, uint32_t item)
{
    using G = EGeo<D, KEY, KR>;
    if (p.use_tma) return (uint32_t)((D / 64) * G::TROWS * 128);  // rows past n arrive as zeros
    const uint32_t bh = fast_div(item, p.div_tiles);
    const int64_t t_first = (int64_t)(item - bh * p.tiles_per_bh) * G::TROWS;
    return (uint32_t)(imin64(G::TROWS, p.n - t_first) * D * 2);
}

// The copies of a tile, completing on `bar` (whose expected bytes the caller
// has already raised by tile_bytes): one tensor copy per 64-column box, or
// one bulk copy per row.  Call from every lane of the warp.
template <int D, bool KEY, int KR = kKeyRows>
__device__ __forceinline__ void issue_copies(const EncodeParams &p, const CUtensorMap &map, uint32_t item,
                                             uint32_t buf, uint32_t bar, int lane)
{
    using G = EGeo<D, KEY, KR>;
    const uint32_t bh = fast_div(item, p.div_tiles);
    const int64_t t_first = (int64_t)(item - bh * p.tiles_per_bh) * G::TROWS;
    const uint32_t b = fast_div(bh, p.div_h), h = bh - b * (uint32_t)p.H;
    if (p.use_tma) {
        if (lane == 0) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_load_4d(buf + c * G::BOX, &map, 64 * c, (int)t_first, (int)h, (int)b, bar);
        }
        return;
    }
    const int rows = (int)imin64(G::TROWS, p.n - t_first);
    if (lane < rows) {
        const uint16_t *src = p.src + b * p.sb + h * p.sh + t_first * p.st;
        for (int row = lane; row < rows; row += 32) bulk_g2s(buf + row * G::RS, src + row * p.st, D * 2, bar);
    }
}

template <int D, bool KEY, int KR = kKeyRows>
__device__ __forceinline__ void issue_tile(const EncodeParams &p, const CUtensorMap &map, uint32_t item, uint32_t buf,
                                           uint32_t bar, int lane)
{
    if (lane == 0) mbar_arrive_expect_tx(bar, tile_bytes<D, KEY, KR>(p, item));
    __syncwarp();
    issue_copies<D, KEY, KR>(p, map, item, buf, bar, lane);
}

// Shared-memory base of a row's 64-column box c and the chunk xor for it.
template <int D, bool KEY, int KR = kKeyRows>
__device__ __forceinline__ uint32_t box_base(const EncodeParams &p, uint32_t buf, int row, int c, uint32_t &xr)
{
    using G = EGeo<D, KEY, KR>;
    xr = p.use_tma ? (uint32_t)(row & 7) : 0u;
    return p.use_tma ? buf + c * G::BOX + row * 128 : buf + row * G::RS + 128 * c;
}

// ------------------------------------------------------------------ packed helpers
__device__ __forceinline__ uint32_t fbits(float f) { return __float_as_uint(f); }

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// RN(x/y) from RN(1/y) (Markstein's correction step; exact for quotients in
// the normal range -- see tests/helpers/markstein_check.c).
__device__ __forceinline__ float ms_div(float x, float y, float ry)
{
    const float q0 = __fmul_rn(x, ry);
    return __fmaf_rn(__fmaf_rn(-y, q0, x), ry, q0);
}

// RN(a*b + c) saturated to [0, 1] (NaN to 0).
__device__ __forceinline__ float ffma_sat(float a, float b, float c)
{
    float d;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// The power of two K with K * den in [2^40, 2^41), for a positive normal den
// below 2^127 (den >= 1e-8 here: exponent field 100..254, K's 40..194).
__device__ __forceinline__ float pow2_scale_for(float den)
{
    const uint32_t e = fbits(den) >> 23;
    return __uint_as_float((294u - e) << 23);
}

// ------------------------------------------------------------------ keys// ------------------------------------------------------------------ keys
// Pack codes given as 0x4B400000 + code (code < 2^BITS) into the BITS-bit
// little-endian stream: accumulate the sums, then subtract what the constant
// 0x4B400000 part contributed (fields do not overlap, so adding is or-ing).
template <int B>
__device__ __forceinline__ void pack_magic(const uint32_t (&m)[32], uint32_t (&w)[B])
{
    constexpr uint32_t M = 0x4B400000u;
    uint32_t corr[B] = {};
#pragma unroll
    for (int k = 0; k < B; ++k) w[k] = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int bit = i * B, word = bit >> 5, off = bit & 31;
        w[word] += m[i] << off;
        corr[word] += M << off;
        if (off + B > 32) {
            w[word + 1] += m[i] >> (32 - off);
            corr[word + 1] += M >> (32 - off);
        }
    }
#pragma unroll
    for (int k = 0; k < B; ++k) w[k] -= corr[k];
}

// The definition step by step (IEEE division), for groups the fast path does
// not cover: NaN/Inf inside, constant groups, scales outside [2^-100, 2^100].
// It reads its 32 keys from the shared tile (a) and writes the group's codes,
// scale and zero point itself.
template <int BITS>
__device__ __noinline__ void key_group_exact(uint32_t a, uint32_t ch0, uint32_t xr, uint8_t *codes, uint16_t *scale_at,
                                             uint16_t *zero_at)
{
    float x[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = lds128(a + 16 * ((ch0 + i) ^ xr));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            x[8 * i + 2 * q] = bf16_lo(u[q]);
            x[8 * i + 2 * q + 1] = bf16_hi(u[q]);
        }
    }
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
    uint32_t code[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        // round, then clip (NaN -> lo, IEEE maxNum/minNum)
        const float c = fminf(fmaxf(rintf(__fsub_rn(__fdiv_rn(x[j], scale), zero)), lo), hi);
        code[j] = (uint32_t)(int)c & ((1u << BITS) - 1u);
    }
    uint32_t out[BITS];
    pack_group<BITS>(code, out);
    store_words<BITS, align_of_bytes(4 * BITS) < 8 ? align_of_bytes(4 * BITS) : 8>(codes, out);
    *scale_at = f32_to_f16_bits(scale);
    *zero_at = f32_to_f16_bits(zero);
}

// Per-group key parameters, computed without branches; ok is false where the
// fast element pass does not apply (NaN/Inf inside, constant or extreme
// groups, max + min overflowing, or a code that would need the clip).
struct KeyParams {
    float scale, rc, zero;
    bool ok;
};

template <int BITS>
__device__ __forceinline__ KeyParams key_params(const uint32_t (&w)[16])
{
    // max propagates NaN (a NaN anywhere takes the exact path); min skips it
    uint32_t a[8], b[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        a[k] = bf16x2_max_nan(w[2 * k], w[2 * k + 1]);
        b[k] = bf16x2_min(w[2 * k], w[2 * k + 1]);
    }
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1)
#pragma unroll
        for (int k = 0; k < s; ++k) {
            a[k] = bf16x2_max_nan(a[k], a[k + s]);
            b[k] = bf16x2_min(b[k], b[k + s]);
        }
    const bool nan = (a[0] & 0x7FFFu) > 0x7F80u || (a[0] & 0x7FFF0000u) > 0x7F800000u;
    const float mx = fmaxf(bf16_lo(a[0]), bf16_hi(a[0])), mn = fminf(bf16_lo(b[0]), bf16_hi(b[0]));
    const float d = __fsub_rn(mx, mn);
    constexpr float C = BITS == 8 ? 254.0f : (float)((1 << BITS) - 1);
    constexpr float RC = BITS == 8 ? 0x1.020408p-8f : BITS == 2 ? 0x1.555556p-2f : BITS == 4 ? 0x1.111112p-4f : 0x1.08421p-5f;
    KeyParams k;
    k.scale = ms_div(d, C, RC);
    k.rc = __frcp_rn(k.scale);
    k.zero = BITS == 8 ? rintf(ms_div(__fadd_rn(mx, mn), 2.0f * k.scale, 0.5f * k.rc)) : rintf(ms_div(mn, k.scale, k.rc));
    // The code RN(RN(x/scale) - zero), rounded, is monotone in x: when the
    // group's min and max land inside [lo, hi], no element needs the clip.
    constexpr float LO = BITS == 8 ? -127.0f : 0.0f, HI = BITS == 8 ? 127.0f : (float)((1 << BITS) - 1);
    const float r_lo = rintf(__fsub_rn(ms_div(mn, k.scale, k.rc), k.zero));
    const float r_hi = rintf(__fsub_rn(ms_div(mx, k.scale, k.rc), k.zero));
    // one branch-free predicate (every comparison is false for NaN)
    k.ok = !nan & (d >= 0x1p-100f) & (d <= 0x1p100f) & (k.scale >= 0x1p-100f) & (k.scale <= 0x1p100f) &
           (fabsf(k.zero) <= 0x1p24f) & (r_lo >= LO) & (r_hi <= HI);
    return k;
}

// idx = round(RN(RN(x/scale) - zero)) for a group that needs no clip: the
// quotient by Markstein's step on fp32 pairs, the rounding by adding 1.5*2^23
// (|value| <= 128 here), so each code sits in the low bits of the sum.
template <int BITS>
__device__ __forceinline__ void key_codes_fast(const uint32_t (&w)[16], const KeyParams &k, uint32_t (&out)[BITS])
{
    const float2 rc2 = make_float2(k.rc, k.rc), ns2 = make_float2(-k.scale, -k.scale), nz2 = make_float2(-k.zero, -k.zero);
    const float2 mg2 = make_float2(12582912.0f, 12582912.0f);
    uint32_t m[32];  // 0x4B400000 + code
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float2 x = make_float2(bf16_lo(w[i]), bf16_hi(w[i]));
        const float2 q0 = __fmul2_rn(x, rc2);
        const float2 q = __ffma2_rn(__ffma2_rn(ns2, q0, x), rc2, q0);
        const float2 c = __fadd2_rn(__fadd2_rn(q, nz2), mg2);
        m[2 * i] = fbits(c.x);
        m[2 * i + 1] = fbits(c.y);
    }
    if constexpr (BITS == 8) {
        // low bytes are the codes in two's complement
#pragma unroll
        for (int i = 0; i < 8; ++i)
            out[i] = __byte_perm(__byte_perm(m[4 * i], m[4 * i + 1], 0x0040), __byte_perm(m[4 * i + 2], m[4 * i + 3], 0x0040),
                                 0x5410);
    } else {
        pack_magic<BITS>(m, out);
    }
}

// A lane's RPL key groups (rows r, r + ROWS, ...): parameters for all first,
// then the element passes, so the groups' dependency chains interleave.
template <int D, int BITS, int KR = kKeyRows>
__device__ __forceinline__ void encode_key_lane(const EncodeParams &p, uint32_t buf, int r, int64_t crow, int part,
                                                int nvalid)
{
    using G = EGeo<D, true, KR>;
    constexpr int R = G::RPL;
    const uint32_t lo = 4 * (part & 1);  // first 16-byte chunk of this lane's 32 keys in the 64-column box
    uint32_t base[R], xr[R];
#pragma unroll
    for (int g = 0; g < R; ++g) base[g] = box_base<D, true, KR>(p, buf, r + g * G::ROWS, part >> 1, xr[g]);
    uint32_t w[R][16];
#pragma unroll
    for (int g = 0; g < R; ++g) {
        if (g < nvalid) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = lds128(base[g] + 16 * ((lo + i) ^ xr[g]));
                w[g][4 * i] = v.x; w[g][4 * i + 1] = v.y; w[g][4 * i + 2] = v.z; w[g][4 * i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[g][i] = 0x3F803F80u;  // 1.0 pairs: a harmless stand-in
        }
    }
    KeyParams kp[R];
    bool all = true;
#pragma unroll
    for (int g = 0; g < R; ++g) {
        kp[g] = key_params<BITS>(w[g]);
        all &= kp[g].ok | (g >= nvalid);
    }
    constexpr int RB = D * BITS / 8, LB = 4 * BITS;
#pragma unroll
    for (int g = 0; g < R; ++g) {
        if (g >= nvalid) break;
        const int64_t row = crow + g * G::ROWS;
        if (!all && !kp[g].ok) {
            key_group_exact<BITS>(base[g], lo, xr[g], p.codes + row * RB + part * LB, p.scale + row * (D / 32) + part,
                                  p.zero + row * (D / 32) + part);
            continue;
        }
        uint32_t out[BITS];
        key_codes_fast<BITS>(w[g], kp[g], out);
        if constexpr (BITS == 8) {
            store_words<8, 16>(p.codes + row * RB + part * LB, out);  // the planes are 16-byte aligned
        } else {
            constexpr int A = align_of_bytes(RB) < align_of_bytes(LB) ? align_of_bytes(RB) : align_of_bytes(LB);
            store_words<BITS, A>(p.codes + row * RB + part * LB, out);
        }
        p.scale[row * (D / 32) + part] = f32_to_f16_bits(kp[g].scale);
        p.zero[row * (D / 32) + part] = f32_to_f16_bits(kp[g].zero);
    }
}

// ------------------------------------------------------------------ values
// number of boundaries strictly below y (searchsorted, side = left); NaN -> 0
template <int BITS>
__device__ __forceinline__ uint32_t value_index(const EncodeParams &p, const float *sbnd, float y)
{
    if constexpr (BITS <= 3) {
        uint32_t k = 0;
#pragma unroll
        for (int i = 0; i < (1 << BITS) - 1; ++i) k += (p.bnd[i] < y) ? 1u : 0u;
        return k;
    } else {
        uint32_t pos = 0;
#pragma unroll
        for (int step = 1 << (BITS - 1); step >= 1; step >>= 1)
            if (sbnd[pos + step - 1] < y) pos += step;
        return pos;
    }
}

template <int BITS>
__device__ __forceinline__ void put_code(uint32_t (&w)[BITS], int j, uint32_t c)
{
    // j is a compile-time index inside unrolled loops; fields do not overlap
    const int bit = j * BITS, word = bit >> 5, off = bit & 31;
    w[word] += c << off;
    if (off + BITS > 32) w[word + 1] += c >> (32 - off);
}

// Value codes of a warp tile are written to a shared staging area (rows x
// row bytes, the tile's own layout in the cache) and leave in one bulk store.
// A lane's 64 value inputs from the shared tile, signs applied.
template <int D>
__device__ __forceinline__ void value_lane_load(uint32_t a, uint32_t xr, uint32_t mtab, int part, bool valid,
                                                float2 (&P)[32])
{
    // P[j] = (element j, element j + 32) of this lane's 64; at head_dim 128 part-1
    // lanes hold them swapped (their two 64-byte halves are read in the other
    // order), for the transform's half-traffic stride-64 stage
    if constexpr (D == 128) xr ^= 4u * (uint32_t)part;
    if (valid) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 u = lds128(a + 16 * (i ^ xr)), v = lds128(a + 16 * ((4 + i) ^ xr));
            const uint32_t uw[4] = {u.x, u.y, u.z, u.w}, vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int k = 4 * i + q;
                // sign masks of elements 2k, 2k+1, 2k+32, 2k+33 (bit 31 set = negate)
                const uint4 m = lds128(mtab + 16 * k);
                P[2 * k] = make_float2(__uint_as_float(uw[q] * 0x10000u + m.x), __uint_as_float(vw[q] * 0x10000u + m.z));
                P[2 * k + 1] = make_float2(__uint_as_float((uw[q] & 0xFFFF0000u) ^ m.y),
                                           __uint_as_float((vw[q] & 0xFFFF0000u) ^ m.w));
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) P[j] = make_float2(0.0f, 0.0f);
    }
}

// Transform, group RMS, indices and packing of a lane's loaded inputs; the
// codes go to the warp's staging area, the scales to the cache.
template <int D, int BITS>
__device__ __forceinline__ void value_lane_codes(const EncodeParams &p, const float *sbnd, float2 (&P)[32],
                                                 uint32_t stage, int64_t crow, int r, int part, bool valid)
{
    using G = EGeo<D, false>;
    // afterwards P[j] holds elements j and j + 32 of the lane's 64 (groups 2 part and
    // 2 part + 1), or at head_dim 128 elements 32 part + j and 64 + 32 part + j
    // (groups part and 2 + part), the second negated on part-1 lanes
    if constexpr (D == 128)
        fwht_pairs_d128<G::ROWS>(P, part);
    else
        fwht_pairs<G::LPR, G::ROWS>(P, part);
    if (!valid) return;
    // y = z / sqrt(d) (the negation undone with it); both groups' sums of squares in element order
    const float c2y = D == 128 && part ? -p.inv_sqrt_d : p.inv_sqrt_d;
    const float2 c2 = make_float2(p.inv_sqrt_d, c2y);
    float2 ss = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        P[j] = __fmul2_rn(P[j], c2);
        ss = __ffma2_rn(P[j], P[j], ss);
    }
    const float2 ms = __fmul2_rn(ss, make_float2(0.03125f, 0.03125f));  // /32, exact
    const float sig0 = __fsqrt_rn(ms.x), sig1 = __fsqrt_rn(ms.y);
    const float den0 = __fadd_rn(sig0, 1e-8f), den1 = __fadd_rn(sig1, 1e-8f);
    uint32_t w0[BITS], w1[BITS];
#pragma unroll
    for (int k = 0; k < BITS; ++k) w0[k] = w1[k] = 0;
    bool done = false;
    if constexpr (BITS <= 4) {
        if (den0 < INFINITY && den1 < INFINITY) {
            // The index counts the boundaries b below y/den.  The table is
            // antisymmetric with b[H-1] = 0, so with m = #{positive b : b*den <
            // |y|} the index is H-1-m for y <= 0 and H+m for y > 0, i.e.
            // 2 idx = 2H-1 + s (2m+1) with s = +1 for y > 0, else -1.
            // b*den < |y| is read off the sign of K^2 (y^2 - (b den)^2), with a
            // per-group power of two K putting K den in [2^40, 2^41): any
            // nonzero value there is at least 2^31 (y^2 has 48 bits, the square
            // of a threshold 24), so saturating to [0, 1] gives exactly 0 or 1.
            // m is found by binary search: at 3 bits the middle threshold picks
            // the outer one to test next, at 4 bits two levels pick the next.
            // It can differ from the division only within a few ulps of a
            // boundary.  The codes are summed as floats, C per chunk weighted
            // 2^(BITS i) (exact: below 2^22 on top of 1.5*2^23), which keeps
            // the bit assembly off the integer pipe.
            constexpr int H = 1 << (BITS - 1);
            constexpr int C = 21 / BITS;            // codes per chunk
            constexpr int NC = (32 + C - 1) / C;    // chunks per group
            const float K0 = pow2_scale_for(den0), K1 = pow2_scale_for(den1);
            float2 nt[H - 1];  // -(K b den)^2 for the positive boundaries
#pragma unroll
            for (int k = 0; k < H - 1; ++k) {
                const float t0 = __fmul_rn(__fmul_rn(p.bnd[H + k], den0), K0);
                const float t1 = __fmul_rn(__fmul_rn(p.bnd[H + k], den1), K1);
                nt[k] = make_float2(-__fmul_rn(t0, t0), -__fmul_rn(t1, t1));
            }
            const float2 nk = make_float2(-K0, -K1), z2 = make_float2(0.0f, 0.0f);
            constexpr float M = 12582912.0f;  // 1.5 * 2^23
            float2 acc[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float wsum = 0.0f;  // (2H - 1) * sum of the chunk's weights, plus M
#pragma unroll
                for (int i = 0; i < C && c * C + i < 32; ++i) wsum += (float)((2 * H - 1) << (BITS * i));
                acc[c] = make_float2(M + wsum, M + wsum);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float2 kv = __ffma2_rn(P[j], nk, z2);  // -K y: sign set iff y > 0 (+0 for y = +-0)
                float2 q;                                    // 2m + 1
                if constexpr (BITS == 4) {
                    // thresholds T1..T7 in nt[0..6]: T4, then T2 or T6, then T1/T3/T5/T7
                    const float2 b1 = make_float2(ffma_sat(kv.x, kv.x, nt[3].x), ffma_sat(kv.y, kv.y, nt[3].y));
                    const float2 n2 = __ffma2_rn(b1, make_float2(nt[5].x - nt[1].x, nt[5].y - nt[1].y), nt[1]);
                    const float2 b2 = make_float2(ffma_sat(kv.x, kv.x, n2.x), ffma_sat(kv.y, kv.y, n2.y));
                    const float2 lo = __ffma2_rn(b1, make_float2(nt[4].x - nt[0].x, nt[4].y - nt[0].y), nt[0]);
                    const float2 hi = __ffma2_rn(b1, make_float2(nt[6].x - nt[2].x, nt[6].y - nt[2].y), nt[2]);
                    const float2 n3 = __ffma2_rn(b2, __fadd2_rn(hi, make_float2(-lo.x, -lo.y)), lo);
                    const float2 b3 = make_float2(ffma_sat(kv.x, kv.x, n3.x), ffma_sat(kv.y, kv.y, n3.y));
                    q = __ffma2_rn(b1, make_float2(8.0f, 8.0f),
                                   __ffma2_rn(b2, make_float2(4.0f, 4.0f),
                                              __ffma2_rn(b3, make_float2(2.0f, 2.0f), make_float2(1.0f, 1.0f))));
                } else if constexpr (BITS == 3) {
                    const float2 b1 = make_float2(ffma_sat(kv.x, kv.x, nt[1].x), ffma_sat(kv.y, kv.y, nt[1].y));
                    const float2 nsel = __ffma2_rn(b1, make_float2(nt[2].x - nt[0].x, nt[2].y - nt[0].y), nt[0]);
                    const float2 b2 = make_float2(ffma_sat(kv.x, kv.x, nsel.x), ffma_sat(kv.y, kv.y, nsel.y));
                    q = __ffma2_rn(b1, make_float2(4.0f, 4.0f), __ffma2_rn(b2, make_float2(2.0f, 2.0f), make_float2(1.0f, 1.0f)));
                } else {
                    const float2 b1 = make_float2(ffma_sat(kv.x, kv.x, nt[0].x), ffma_sat(kv.y, kv.y, nt[0].y));
                    q = __ffma2_rn(b1, make_float2(2.0f, 2.0f), make_float2(1.0f, 1.0f));
                }
                // s (2m + 1): negative unless y > 0
                const float2 sq = make_float2(__uint_as_float(fbits(q.x) | (~fbits(kv.x) & 0x80000000u)),
                                              __uint_as_float(fbits(q.y) | (~fbits(kv.y) & 0x80000000u)));
                const float wj = (float)(1u << (BITS * (j % C)));
                acc[j / C] = __ffma2_rn(sq, make_float2(wj, wj), acc[j / C]);
            }
            // chunk c holds 2 x (codes 7c.. as a C*BITS-bit string) in its low 22 bits; place it at bit C*BITS*c
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const uint32_t u0 = fbits(acc[c].x) & 0x3FFFFFu, u1 = fbits(acc[c].y) & 0x3FFFFFu;
                const int bit = c * C * BITS, word = bit >> 5, off = bit & 31;
                const int nbits = (32 - c * C < C ? 32 - c * C : C) * BITS;
                if (off == 0) {
                    w0[word] += u0 >> 1;
                    w1[word] += u1 >> 1;
                } else {
                    w0[word] += u0 << (off - 1);
                    w1[word] += u1 << (off - 1);
                }
                if (off + nbits > 32) {
                    w0[word + 1] += u0 >> (33 - off);
                    w1[word + 1] += u1 >> (33 - off);
                }
            }
            done = true;
        }
    }
    if (!done) {
        const bool fin0 = den0 < INFINITY, fin1 = den1 < INFINITY;
        const float r0 = __frcp_rn(den0), r1 = __frcp_rn(den1);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            // finite rows: y * RN(1/den), within an ulp of the quotient; others the definition's division
            const float q0 = fin0 ? __fmul_rn(P[j].x, r0) : __fdiv_rn(P[j].x, den0);
            const float q1 = fin1 ? __fmul_rn(P[j].y, r1) : __fdiv_rn(P[j].y, den1);
            put_code<BITS>(w0, j, value_index<BITS>(p, sbnd, q0));
            put_code<BITS>(w1, j, value_index<BITS>(p, sbnd, q1));
        }
    }
    if constexpr (D == 128) {
        // groups part and 2 + part of the row: 4 BITS bytes of codes and one fp16 scale each
        constexpr int RB = D * BITS / 8, GB = 4 * BITS;
        const uint32_t ax = stage + r * RB + part * GB, ay = ax + 2 * GB;
#pragma unroll
        for (int k = 0; k < BITS; ++k) {
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(ax + 4 * k), "r"(w0[k]) : "memory");
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(ay + 4 * k), "r"(w1[k]) : "memory");
        }
        p.scale[crow * (D / 32) + part] = f32_to_f16_bits(sig0);
        p.scale[crow * (D / 32) + 2 + part] = f32_to_f16_bits(sig1);
    } else {
        uint32_t w[2 * BITS];
#pragma unroll
        for (int k = 0; k < BITS; ++k) {
            w[k] = w0[k];
            w[BITS + k] = w1[k];
        }
        constexpr int RB = D * BITS / 8, LB = 8 * BITS;
        constexpr int A = align_of_bytes(LB) < 8 ? align_of_bytes(LB) : 8;
        const uint32_t at = stage + r * RB + part * LB;
#pragma unroll
        for (int i = 0; i < 2 * BITS; i += A / 4) {
            if constexpr (A == 8)
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(at + 4 * i), "r"(w[i]), "r"(w[i + 1]) : "memory");
            else
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(at + 4 * i), "r"(w[i]) : "memory");
        }
        const uint32_t sw = (uint32_t)f32_to_f16_bits(sig0) | ((uint32_t)f32_to_f16_bits(sig1) << 16);
        *reinterpret_cast<uint32_t *>(p.scale + crow * (D / 32) + 2 * part) = sw;
    }
}

template <int D, int BITS>
__device__ __forceinline__ void encode_value_lane(const EncodeParams &p, const float *sbnd, uint32_t a, uint32_t xr,
                                                  uint32_t mtab, uint32_t stage, int64_t crow, int r, int part, bool valid)
{
    float2 P[32];
    value_lane_load<D>(a, xr, mtab, part, valid, P);
    value_lane_codes<D, BITS>(p, sbnd, P, stage, crow, r, part, valid);
}

// ------------------------------------------------------------------ kernels
// The work of CTA `cta` of `ncta` encoding keys (KEY) or values.
template <int D, int BITS, bool KEY>
__device__ __forceinline__ void encode_body(const EncodeParams &p, const CUtensorMap &map, uint8_t *smem_raw,
                                            uint32_t cta, uint32_t ncta)
{
    using G = EGeo<D, KEY>;
    constexpr int SB = (!KEY && BITS > 3) ? 1024 : 0;
    // tiles need 1024-byte alignment (swizzle atoms); the rest follows them
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int STG = KEY ? 0 : VStage<D, BITS>::BYTES;
    uint8_t *tiles = smem;
    uint8_t *rest = tiles + kWarps * 2 * G::TILE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(rest);  // 2 per warp
    float *sbnd = reinterpret_cast<float *>(rest + 16 * kWarps);
    uint8_t *mtab = rest + 16 * kWarps + SB;
    uint8_t *stages = mtab + G::MTAB;  // value code staging, one per warp
    const uint32_t buf0 = smem_addr(tiles + warp * 2 * G::TILE), buf1 = buf0 + G::TILE;
    const uint32_t bar0 = smem_addr(&bars[2 * warp]), bar1 = bar0 + 8;

    if constexpr (SB > 0) {
        for (int i = threadIdx.x; i < (1 << BITS) - 1; i += blockDim.x) sbnd[i] = p.bnd[i];
    }
    if constexpr (!KEY) {
        // sign masks: entry (part, k) = elements 64 part + {2k, 2k+1, 2k+32, 2k+33}
        for (int i = threadIdx.x; i < G::LPR * 16; i += blockDim.x) {
            const int part = i >> 4, k = i & 15;
            // at head_dim 128 part-1 lanes hold swapped pairs (element j + 32, element j)
            const int e = 64 * part + 2 * k + (D == 128 && part ? 32 : 0), f = D == 128 && part ? e - 32 : e + 32;
            const uint4 m = make_uint4(sign_negative(p.sg, e) ? 0x80000000u : 0u, sign_negative(p.sg, e + 1) ? 0x80000000u : 0u,
                                       sign_negative(p.sg, f) ? 0x80000000u : 0u, sign_negative(p.sg, f + 1) ? 0x80000000u : 0u);
            *reinterpret_cast<uint4 *>(mtab + part * 272 + 16 * k) = m;
        }
    }
    if (lane == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar1, 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int r = lane % G::ROWS, part = lane / G::ROWS;
    const uint32_t my_mtab = smem_addr(mtab) + part * 272;
    const uint32_t W = ncta * kWarps;
    uint32_t item = cta * kWarps + warp;
    if (item < p.items) issue_tile<D, KEY>(p, map, item, buf0, bar0, lane);
    for (uint32_t k = 0; item < p.items; item += W, ++k) {
        const uint32_t next = item + W;
        const uint32_t buf = (k & 1) ? buf1 : buf0, bar = (k & 1) ? bar1 : bar0;
        if (next < p.items) issue_tile<D, KEY>(p, map, next, (k & 1) ? buf0 : buf1, (k & 1) ? bar0 : bar1, lane);
        if (!mbar_wait_bounded(bar, (k >> 1) & 1, p.err)) {
            // give the other copy a bounded chance to land before leaving
            if (next < p.items) mbar_wait_bounded((k & 1) ? bar0 : bar1, ((k + 1) >> 1) & 1, p.err);
            if (!KEY && lane == 0) bulk_wait0();
            return;
        }
        const uint32_t bh = fast_div(item, p.div_tiles);
        const int64_t t_first = (int64_t)(item - bh * p.tiles_per_bh) * G::TROWS;
        const bool valid = t_first + r < p.n;
        const int64_t crow = (int64_t)bh * p.cap + p.t0 + t_first + r;
        if constexpr (KEY) {
            // rows r, r + ROWS, ... of the tile that exist
            const int nvalid = (int)imin64(G::RPL, (p.n - t_first - r + G::ROWS - 1) / G::ROWS);
            if (valid) encode_key_lane<D, BITS>(p, buf, r, crow, part, nvalid);
        } else {
            constexpr int RB = VStage<D, BITS>::RB;
            const uint32_t stage = smem_addr(stages + warp * STG);
            // the previous tile's bulk store must have read the staging area
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
            // every lane of a row joins the cross-lane stages, so no early exit
            uint32_t xr;
            const uint32_t a = box_base<D, false>(p, buf, r, part, xr);
            encode_value_lane<D, BITS>(p, sbnd, a, xr, my_mtab, stage, crow, r, part, valid);
            fence_proxy_async_smem();
            __syncwarp();
            const int rows = (int)imin64(G::TROWS, p.n - t_first);
            uint8_t *dst = p.codes + (crow - r) * RB;
            if (((uintptr_t)dst & 15) == 0 && (rows * RB) % 16 == 0) {
                if (lane == 0) {
                    bulk_s2g(dst, stage, (uint32_t)(rows * RB));
                    bulk_commit();
                }
            } else {
                // destination or size not a multiple of 16 bytes (row bytes are a multiple of 8): plain stores
                for (int i = 8 * lane; i < rows * RB; i += 256)
                    *reinterpret_cast<uint2 *>(dst + i) = *reinterpret_cast<const uint2 *>(stages + warp * STG + i);
            }
        }
        __syncwarp();
    }
    // staged value codes: the bulk stores must have read shared memory before the CTA ends
    if (!KEY && lane == 0) bulk_wait0();
}

// Every launch of this library is a programmatic dependent of the kernel
// before it on the stream and waits for that kernel before touching memory.
// The exception is the value launch of an append made of two launches (keys,
// then values): it touches none of the key planes, so it starts as soon as
// the key kernel has started and takes the SMs that key CTAs leave in their
// last round; it waits for the key grid only before it ends, which keeps
// stream order for whatever is queued after the append.
template <int D, int BITS, bool KEY>
__global__ void __launch_bounds__(kWarps * 32)
    encode_kernel(const __grid_constant__ EncodeParams p, const __grid_constant__ CUtensorMap map)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    if constexpr (KEY) pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    encode_body<D, BITS, KEY>(p, map, smem_raw, blockIdx.x, gridDim.x);
    if constexpr (!KEY) pdl_wait_primary();
}

// Keys and values in one launch: CTAs [0, key_ctas) encode the keys, the
// others the values (see run_kv for how the CTAs are shared out).
template <int D, int KB, int VB>
__global__ void __launch_bounds__(kWarps * 32)
    encode_kv_kernel(const __grid_constant__ EncodeParams pk, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ EncodeParams pv, const __grid_constant__ CUtensorMap mv, uint32_t key_ctas)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    if (blockIdx.x < key_ctas)
        encode_body<D, KB, true>(pk, mk, smem_raw, blockIdx.x, key_ctas);
    else
        encode_body<D, VB, false>(pv, mv, smem_raw, blockIdx.x - key_ctas, gridDim.x - key_ctas);
}

// dynamic shared memory of encode_body<D, BITS, KEY>
template <int D, int BITS, bool KEY>
constexpr size_t encode_smem()
{
    using G = EGeo<D, KEY>;
    return 1024 /*alignment slack*/ + (size_t)kWarps * 2 * G::TILE + 16 * kWarps + ((!KEY && BITS > 3) ? 1024 : 0) +
           G::MTAB + (size_t)kWarps * (KEY ? 0 : VStage<D, BITS>::BYTES);
}

// A value launch must directly follow the key launch of the same append.
template <int D, int BITS, bool KEY>
cudaError_t run(const EncodeParams &p, const CUtensorMap &map, cudaStream_t s)
{
    const size_t smem = encode_smem<D, BITS, KEY>();
    auto kern = encode_kernel<D, BITS, KEY>;
    static int per_sm = 0;  // same on every GB300; only a successful query is kept
    if (!per_sm) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kWarps * 32, smem);
        if (e != cudaSuccess) return e;
        per_sm = n > 0 ? n : 1;
    }
    const int64_t want = ((int64_t)p.items + kWarps - 1) / kWarps;
    const int grid = (int)imin64(want, (int64_t)num_sms() * per_sm);
    return launch_dependent(kern, dim3((unsigned)grid), dim3(kWarps * 32), smem, s, p, map);
}

// Keys and values of a small append in one launch (encode_kv_kernel), every
// CTA resident at once.
template <int D, int KB, int VB>
cudaError_t run_kv(const EncodeParams &pk, const CUtensorMap &mk, const EncodeParams &pv, const CUtensorMap &mv,
                   uint32_t key_ctas, uint32_t value_ctas, cudaStream_t s)
{
    constexpr size_t sk = encode_smem<D, KB, true>(), sv = encode_smem<D, VB, false>();
    constexpr size_t smem = sk > sv ? sk : sv;
    auto kern = encode_kv_kernel<D, KB, VB>;
    static bool attr = false;  // same on every GB300; only a successful call is kept
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    return launch_dependent(kern, dim3(key_ctas + value_ctas), dim3(kWarps * 32), smem, s, pk, mk, pv, mv, key_ctas);
}

template <int D>
cudaError_t dispatch_key(int kb, const EncodeParams &p, const CUtensorMap &map, cudaStream_t s)
{
    switch (kb) {
    case 2: return run<D, 2, true>(p, map, s);
    case 4: return run<D, 4, true>(p, map, s);
    case 5: return run<D, 5, true>(p, map, s);
    case 8: return run<D, 8, true>(p, map, s);
    }
    return cudaErrorInvalidValue;
}

template <int D>
cudaError_t dispatch_value(int vb, const EncodeParams &p, const CUtensorMap &map, cudaStream_t s)
{
    switch (vb) {
    case 2: return run<D, 2, false>(p, map, s);
    case 3: return run<D, 3, false>(p, map, s);
    case 4: return run<D, 4, false>(p, map, s);
    case 5: return run<D, 5, false>(p, map, s);
    case 8: return run<D, 8, false>(p, map, s);
    }
    return cudaErrorInvalidValue;
}

// Tensor map over the [B][H][n][D] bf16 input (any strides the API accepts):
// boxes of 64 columns x rows, 128-byte swizzle.  False if the driver refuses
// it (the kernels then copy row by row).
inline bool input_map(CUtensorMap *map, const uint16_t *src, int D, int64_t n, int H, int B, const int64_t st[3],
                      int rows)
{
    auto fn = tensor_map_encoder();
    if (!fn || n >= (int64_t(1) << 31)) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)n, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)rows, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(src), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tiles of `rows` token rows per (sequence, kv-head); false if the count
// does not fit the kernels' 31-bit item index.
inline bool set_items(EncodeParams &p, int64_t n, int rows, const CacheView &c)
{
    const int64_t tiles = (n + rows - 1) / rows, items = tiles * (int64_t)c.B * c.H;
    if (items >= (int64_t(1) << 31)) return false;
    p.tiles_per_bh = (uint32_t)tiles;
    p.items = (uint32_t)items;
    p.div_tiles = make_fastdiv(tiles > 0 ? (uint32_t)tiles : 1u);
    return true;
}

template <int D>
cudaError_t encode_d(const CacheView &c, const uint16_t *k, const int64_t ks[3], const uint16_t *v,
                     const int64_t vs[3], int64_t t0, int64_t n, cudaStream_t s)
{
    EncodeParams p{};
    p.H = c.H;
    p.cap = c.cap;
    p.t0 = t0;
    p.n = n;
    p.inv_sqrt_d = inv_sqrt_head_dim(D);
    p.sg = c.signs;
    p.err = device_error_word();
    if (!p.err) return cudaErrorInvalidDevice;
    const Tables &tab = codebook_tables(c.vb);
    for (int i = 0; i < (1 << c.vb) - 1; ++i) p.bnd[i] = tab.boundaries[i];

    EncodeParams pk = p, pv = p;
    CUtensorMap mk{}, mv{};
    pk.src = k;
    pk.sb = ks[0]; pk.sh = ks[1]; pk.st = ks[2];
    pk.codes = c.k_codes;
    pk.scale = c.k_scale;
    pk.zero = c.k_zero;
    pk.div_h = make_fastdiv((uint32_t)c.H);
    if (!set_items(pk, n, EGeo<D, true>::TROWS, c)) return cudaErrorInvalidValue;
    pk.use_tma = input_map(&mk, k, D, n, c.H, c.B, ks, EGeo<D, true>::TROWS) ? 1 : 0;

    pv.src = v;
    pv.sb = vs[0]; pv.sh = vs[1]; pv.st = vs[2];
    pv.codes = c.v_codes;
    pv.scale = c.v_scale;
    pv.zero = nullptr;
    pv.div_h = make_fastdiv((uint32_t)c.H);
    if (!set_items(pv, n, EGeo<D, false>::TROWS, c)) return cudaErrorInvalidValue;
    pv.use_tma = input_map(&mv, v, D, n, c.H, c.B, vs, EGeo<D, false>::TROWS) ? 1 : 0;

    // a small append (a few rows per sequence-head, as in a decode step) runs
    // keys and values in one launch when both grids fit one CTA per SM; a
    // larger one as two launches (keys, then values)
    const uint32_t gk = (pk.items + kWarps - 1) / kWarps, gv = (pv.items + kWarps - 1) / kWarps;
    if ((int64_t)gk + gv <= num_sms() && c.vb == 3 && (c.kb == 8 || c.kb == 4)) {
        if (c.kb == 8) return run_kv<D, 8, 3>(pk, mk, pv, mv, gk, gv, s);
        return run_kv<D, 4, 3>(pk, mk, pv, mv, gk, gv, s);
    }
    cudaError_t e = dispatch_key<D>(c.kb, pk, mk, s);
    if (e != cudaSuccess) return e;
    return dispatch_value<D>(c.vb, pv, mv, s);
}

}  // namespace
}  // namespace tq
