// tq_attention_generic.cuh -- fused dequantise-on-fetch attention for every
// head_dim, bit pair and GQA group size, with one or several query rows per
// sequence.  The kernel in tq_attention.cu is the specialised one-row path for
// head_dims 64, 128 and 256, 8- or 4-bit keys, 2-, 3- or 4-bit values and
// groups of 8 q-heads; this one covers the rest with the same method and the
// same tolerance.
//
// Method: mlx-bun "TurboQuant -- rotation-based quantization", Part A:
// "Architecture in mlx-bun" (attention reads the dequantised window),
// "Algorithm" (key (code + zero) * scale, value centroid[code] * rms),
// "Deferred inverse FWHT" (the weighted sum is formed in the rotated domain
// and un-rotated once per query row), and "Packed-value decode fusion
// investigation" (forward passes that append M = 1, 4 or 128 rows and attend
// to the cache including them: query row i of M sees the rows before
// seq_len - M + i + 1).
//
// Design, after the specialised kernel's: split-KV CTAs stream 64-token stages
// through a 2-deep shared-memory ring (bulk copies completing on an mbarrier;
// the last warp to finish a stage refills it); each of the 2 warps takes two
// 16-token tiles and works on both inside every group iteration, with one
// softmax step over both (4 warps of one tile at head_dim 512).  QK^T and PV
// run on mma.sync m16n8k16 (f16 in, f32 accumulate).
// The MMA's N runs over "columns", a column being one (query row, q-head) of
// the kv-head's G * M; a CTA takes NB blocks of 8 columns (NB = 1, 2 or 4 by
// head_dim), so each dequantised key and value fragment feeds NB MMAs and a
// kv-head whose columns fit in one CTA reads its cache rows once.  More
// columns use several CTAs (column blocks); unused columns are masked.  Key
// codes enter the MMA as exact f16 integers (1024 + code) and the per-group
// affine is applied to the scores; value codes are looked up in an f16
// centroid table and the rms is folded into P.  8- and 4-bit keys and 3- and
// 2-bit values have their own instantiations (constant shifts, lookups by byte
// permute); other widths are run-time values, cut from the packed rows with
// funnel shifts.  Each head_dim's kernels compile in their own translation
// unit (tq_attention_generic_d<head_dim>.cu).
#pragma once
#include <cuda.h>

#include "tq_common.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int gT = 64;              // tokens per stage
constexpr int gN = 8;               // q-heads per CTA (the MMA's N)
constexpr int gMaxStages = 3;

struct GenParams {
    const uint8_t *k_codes, *v_codes;
    const uint16_t *k_scale, *k_zero, *v_scale;
    const uint16_t *q;  // [B][M][QH][D] bf16
    float *part_o;      // [B][H][HB][S][CB][D]
    float *part_ml;     // [B][H][HB][S][CB][2]
    uint32_t *err;
    int H, QH, G, M, cols, HB, splits, kb, vb, stages;  // cols = G * M columns per kv-head
    int64_t cap, seq_len, tokens_per_split;
    int64_t base0;                                 // seq_len - M + 1: query row i sees rows [0, base0 + i)
    int rbk, rbv;                                  // packed row bytes of keys and values
    // ring layout: the key tiles of all slots (key_bytes each, 1024-byte multiples
    // for swizzled tiles), then the other planes of all slots (stage_bytes each,
    // at offsets off_ks .. off_v)
    int off_ks, off_kz, off_vs, off_v, stage_bytes, key_bytes;
    float scale_log2, koff;                        // softmax scale * log2(e); f16 offset of a key code
    uint16_t cen[256];                             // value centroids as f16 bits
};

__device__ __forceinline__ void g_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t g_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t g_pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t g_hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float g_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t g_lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t g_lds8(uint32_t a)
{
    uint16_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t g_lds16(uint32_t a)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint2 g_lds64(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ void g_tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Key codes of dims 32G + 8c .. +7 of one packed row -> four f16x2 pairs
// (dims 2p, 2p+1), each half koff + code with koff = 1024 (unsigned codes) or
// 1152 (int8 codes, stored offset by 128).  KEY 8 and 4: the 8 codes are one
// aligned 64- or 32-bit word (constant shifts); KEY 0: kb bits a code, cut
// from a 64-bit window.
template <int KEY>
__device__ __forceinline__ void key_pairs(uint32_t row, int G, int c, int kb, uint32_t (&pr)[4])
{
    if constexpr (KEY == 8) {
        const uint2 w = g_lds64(row + (4 * G + c) * 8);
        const uint32_t l = w.x ^ 0x80808080u, h = w.y ^ 0x80808080u;  // int8 -> code + 128
        pr[0] = __byte_perm(l, 0x64646464u, 0x5140);
        pr[1] = __byte_perm(l, 0x64646464u, 0x5342);
        pr[2] = __byte_perm(h, 0x64646464u, 0x5140);
        pr[3] = __byte_perm(h, 0x64646464u, 0x5342);
    } else if constexpr (KEY == 4) {
        const uint32_t x = g_lds32(row + (4 * G + c) * 4);  // codes k at bits 4k
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t t = x >> (8 * p);  // codes 2p, 2p+1 at bits 0-3, 4-7
            pr[p] = ((t & 0x0Fu) | ((t << 12) & 0x000F0000u)) | 0x64006400u;
        }
    } else {
        const int off = (4 * G + c) * kb;  // byte offset of the 8 codes (8 * kb bits)
        const uint32_t a = row + (off & ~3);
        const uint32_t lo = g_lds32(a), hi = g_lds32(a + 4);
        const uint64_t v = ((uint64_t)hi << 32 | lo) >> ((off & 3) * 8);
        const uint32_t mask = (1u << kb) - 1u;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t c0 = (uint32_t)(v >> (2 * p * kb)) & mask, c1 = (uint32_t)(v >> ((2 * p + 1) * kb)) & mask;
            pr[p] = (c0 | (c1 << 16)) | 0x64006400u;
        }
    }
}

// 8- and 4-bit key tiles arrive by tensor copies with a shared-memory swizzle:
// boxes of BOXB bytes (32, 64 or 128, the row or a 128-byte slice of it) x
// gT rows, the 16-byte chunk index of a row xor-ed with row bits, so the
// rows a half-warp reads in one fragment load fall on different banks.
template <int D, int KEY>
struct KSwz {
    static constexpr int RB = D * KEY / 8;
    static constexpr int BOXB = RB < 128 ? RB : 128;
    static constexpr int NBOX = RB / BOXB;
};

// Shared address of byte `off` of stage row r of a swizzled key tile.
template <int D, int KEY>
__device__ __forceinline__ uint32_t ksw_addr(uint32_t st, int r, int off)
{
    using K = KSwz<D, KEY>;
    const int box = off / K::BOXB, col = off % K::BOXB;
    const int x = K::BOXB == 128 ? (r & 7) : K::BOXB == 64 ? ((r >> 1) & 3) : ((r >> 2) & 1);
    return st + box * (gT * K::BOXB) + r * K::BOXB + ((((col >> 4) ^ x)) << 4) + (col & 15);
}

// The key pairs of key_pairs<8> / <4> from a swizzled tile.
template <int D, int KEY>
__device__ __forceinline__ void key_pairs_sw(uint32_t st, int r, int G, int c, uint32_t (&pr)[4])
{
    if constexpr (KEY == 8) {
        const uint2 w = g_lds64(ksw_addr<D, 8>(st, r, (4 * G + c) * 8));
        const uint32_t l = w.x ^ 0x80808080u, h = w.y ^ 0x80808080u;  // int8 -> code + 128
        pr[0] = __byte_perm(l, 0x64646464u, 0x5140);
        pr[1] = __byte_perm(l, 0x64646464u, 0x5342);
        pr[2] = __byte_perm(h, 0x64646464u, 0x5140);
        pr[3] = __byte_perm(h, 0x64646464u, 0x5342);
    } else {
        // codes k at bits 4k; pair p = codes (p, p + 4) as f16 (1024 + code), one
        // logic op after a shift (the q fragments of 4-bit instantiations hold
        // the dims in that order)
        const uint32_t x = g_lds32(ksw_addr<D, 4>(st, r, (4 * G + c) * 4));
#pragma unroll
        for (int p = 0; p < 4; ++p) pr[p] = ((x >> (4 * p)) & 0x000F000Fu) | 0x64006400u;
    }
}

// Value codes of dims 32G + 4g .. +3 of one packed row -> their f16 centroids.
__device__ __forceinline__ void value_quad(uint32_t row, int G, int g, int vb, uint32_t lut, uint32_t (&h)[4])
{
    const int b = (32 * G + 4 * g) * vb;
    const uint32_t a = row + 4 * (b >> 5);
    const uint32_t x = __funnelshift_r(g_lds32(a), g_lds32(a + 4), b & 31);
    const uint32_t mask = (1u << vb) - 1u;
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = g_lds16(lut + 2 * ((x >> (k * vb)) & mask));
}

template <int D, int NB>
struct GGeo {
    static constexpr int NG = D / 32;
    static constexpr int KS = D / 16;                       // k-steps of QK^T, m-tiles of PV
    static constexpr int CB = gN * NB;                      // columns per CTA
    // q fragments: [column][k-step][c] x (b0, b1), columns QCOL bytes apart: the
    // 32-byte pad puts the 4 columns a half-warp reads on different banks
    static constexpr int QCOL = KS * 4 * 8 + 32;
    static constexpr int QF = CB * QCOL;
    static constexpr int QS = (NG + 1) * CB * 4;            // group sums of the f16 q, then per-column score scale
    // warps per CTA and 16-row tiles per warp and stage (worked on together): 2 x 2,
    // except at head_dim 512, whose registers and stage ring leave room for two CTAs
    // per SM, where 4 warps of one tile each keep 8 warps resident
    static constexpr int W = D >= 512 ? 4 : 2, TILES = D >= 512 ? 1 : 2, THREADS = 32 * W;
    static constexpr int MERGE = W * CB * (D + 2) * 4;      // per-warp partials (reuse the ring)
    // resident CTAs per SM the register budget is sized for: the output
    // accumulators take D * NB / 4 registers a thread
    static constexpr int MIN_BLOCKS = D >= 512 ? 1 : (D * NB / 4 <= 32 ? 6 : 4);
};

// VLUT: how value codes become f16 centroids.  0: a shared-memory table; 3 or
// 2: 3- or 2-bit values looked up with byte permutes in registers.  KEY: how
// key codes are cut (key_pairs).  Separate instantiations: the same choices made
// at run time inside one kernel cost more than they saved (the larger unrolled
// body).
template <int D, int NB, int VLUT, int KEY>
__global__ void __launch_bounds__(GGeo<D, NB>::THREADS, GGeo<D, NB>::MIN_BLOCKS)
    attn_generic_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ GenParams p)
{
    using A = GGeo<D, NB>;
    constexpr int CB = A::CB;
    pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment: swizzled key boxes start on a swizzle atom
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int ring_bytes = p.stages * (p.key_bytes + p.stage_bytes);
    const int ring = ring_bytes > A::MERGE ? ring_bytes : A::MERGE;
    uint8_t *stages = smem;
    float *merge = reinterpret_cast<float *>(smem);
    uint8_t *qf = smem + ring;
    float *qsum = reinterpret_cast<float *>(qf + A::QF);
    // the f16 centroid table in shared memory serves VLUT 0 only (the others
    // look centroids up in registers)
    uint16_t *lut = reinterpret_cast<uint16_t *>(qf + A::QF + A::QS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(qf + A::QF + A::QS + (VLUT == 0 ? 512 : 0));
    uint32_t *done = reinterpret_cast<uint32_t *>(bars + gMaxStages);
    const uint32_t full0 = smem_addr(bars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, h = blockIdx.y / p.HB, hb = blockIdx.y - h * p.HB, b = blockIdx.z;
    const int64_t bh = (int64_t)b * p.H + h;
    // columns col0 .. col0 + CB - 1; column col is query row col / G, q-head
    // h G + col % G; query row i sees cache rows [0, base0 + i)
    const int col0 = hb * CB;
    const int col_last = (p.cols < col0 + CB ? p.cols : col0 + CB) - 1;
    const int64_t lim_lo = p.base0 + col0 / p.G, lim_hi = p.base0 + col_last / p.G;
    const int64_t t_begin = (int64_t)split * p.tokens_per_split;
    const int64_t t_end = imin64(lim_hi, t_begin + p.tokens_per_split);
    const int n_stages = t_end > t_begin ? (int)((t_end - t_begin + gT - 1) / gT) : 0;
    const int NG = D / 32;

    auto issue = [&](int s) {
        const int slot = s % p.stages;
        const int64_t t = t_begin + (int64_t)s * gT;
        const int rows = (int)imin64(gT, p.cap - t);
        const int64_t row0 = bh * p.cap + t;
        const uint32_t kst = smem_addr(stages + slot * p.key_bytes), bar = full0 + 8 * slot;
        const uint32_t st = smem_addr(stages + p.stages * p.key_bytes + slot * p.stage_bytes);
        if constexpr (KEY != 0) {
            // key rows by tensor copies (whole boxes; rows past the cache arrive as zeros)
            using K = KSwz<D, KEY>;
            mbar_arrive_expect_tx(bar, (uint32_t)(gT * K::RB + rows * (p.rbv + 3 * NG * 2)));
#pragma unroll
            for (int j = 0; j < K::NBOX; ++j)
                g_tma_2d(kst + j * gT * K::BOXB, &kmap, j * K::BOXB, (int)row0, bar);
        } else {
            mbar_arrive_expect_tx(bar, (uint32_t)(rows * (p.rbk + p.rbv + 3 * NG * 2)));
            bulk_g2s(kst, p.k_codes + row0 * p.rbk, rows * p.rbk, bar);
        }
        bulk_g2s(st + p.off_ks, p.k_scale + row0 * NG, rows * NG * 2, bar);
        bulk_g2s(st + p.off_kz, p.k_zero + row0 * NG, rows * NG * 2, bar);
        bulk_g2s(st + p.off_vs, p.v_scale + row0 * NG, rows * NG * 2, bar);
        bulk_g2s(st + p.off_v, p.v_codes + row0 * p.rbv, rows * p.rbv, bar);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            done[s] = 0;
        }
        fence_mbar_init();
        for (int s = 0; s < p.stages && s < n_stages; ++s) issue(s);
    }
    if constexpr (VLUT == 0)
        for (int i = threadIdx.x; i < (1 << p.vb); i += blockDim.x) lut[i] = p.cen[i];

    // ---------------------------------------------------------------- q of the CTA's columns
    // Per block of 8 columns, warp w prepares columns 2w, 2w+1; lane l holds
    // dims 4 (l % 16) + 64 j + {0..3} of column 2w + l / 16.  Each column is
    // scaled by a power of two so its largest |q| lands in [2^14, 2^15) before
    // the f16 rounding; columns past the last are zero.
#pragma unroll 1
    for (int u = warp; u < NB * (gN / 2); u += A::W) {
        const int n = (u / (gN / 2)) * gN + 2 * (u % (gN / 2)) + (lane >> 4), l16 = lane & 15;
        const int col = col0 + n;
        const bool real = col < p.cols;
        const int qi = real ? col / p.G : 0, qw = real ? col - qi * p.G : 0;
        const uint16_t *qrow = p.q + (((int64_t)b * p.M + qi) * p.QH + (int64_t)h * p.G + qw) * D;
        float qv[D / 64][4];
        float mx = 0.0f;
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
            uint2 w = make_uint2(0u, 0u);
            if (real) w = *reinterpret_cast<const uint2 *>(qrow + 64 * j + 4 * l16);
            qv[j][0] = bf16_lo(w.x); qv[j][1] = bf16_hi(w.x); qv[j][2] = bf16_lo(w.y); qv[j][3] = bf16_hi(w.y);
#pragma unroll
            for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fabsf(qv[j][i]));
        }
#pragma unroll
        for (int m = 1; m < 16; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        int e = 0;
        if (mx > 0.0f && mx < INFINITY) e = 14 - (((int)(__float_as_uint(mx) >> 23) & 0xFF) - 127);
        e = e < -100 ? -100 : (e > 100 ? 100 : e);
        const float qscale = ldexpf(1.0f, e);
        // dims 64j + 4 l16 + {0..3} lie in group G = 2j + l16 / 8 at offset 4 (l16 % 8);
        // fragment slot (k-step 2G + jj, c, b0/b1) holds dims 8c + 4jj + {0,1} / {2,3}
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
            const int G = 2 * j + (l16 >> 3), o = 4 * (l16 & 7), c = o >> 3, jj = (o >> 2) & 1;
            float f[4];
            uint32_t hw[2];
            hw[0] = g_pack_f16x2(qv[j][0] * qscale, qv[j][1] * qscale);
            hw[1] = g_pack_f16x2(qv[j][2] * qscale, qv[j][3] * qscale);
            f[0] = __low2float(*reinterpret_cast<__half2 *>(&hw[0]));
            f[1] = __high2float(*reinterpret_cast<__half2 *>(&hw[0]));
            f[2] = __low2float(*reinterpret_cast<__half2 *>(&hw[1]));
            f[3] = __high2float(*reinterpret_cast<__half2 *>(&hw[1]));
            uint32_t *slot = reinterpret_cast<uint32_t *>(qf + n * A::QCOL + ((2 * G + jj) * 4 + c) * 8);
            if constexpr (KEY == 4) {
                // dims 8c + {0..3} (jj = 0) and 8c + {4..7} (jj = 1) sit in neighbouring
                // lanes; the 4-bit key pairs are (k, k + 4), so k-step jj = 0 takes
                // (8c, 8c+4), (8c+1, 8c+5) and jj = 1 takes (8c+2, 8c+6), (8c+3, 8c+7)
                const uint32_t o0 = __shfl_xor_sync(0xffffffffu, hw[0], 1), o1 = __shfl_xor_sync(0xffffffffu, hw[1], 1);
                if (jj == 0) {
                    slot[0] = __byte_perm(hw[0], o0, 0x5410);  // (own 8c, partner 8c+4)
                    slot[1] = __byte_perm(hw[0], o0, 0x7632);  // (8c+1, 8c+5)
                } else {
                    slot[0] = __byte_perm(o1, hw[1], 0x5410);  // (partner 8c+2, own 8c+6)
                    slot[1] = __byte_perm(o1, hw[1], 0x7632);  // (8c+3, 8c+7)
                }
            } else {
                slot[0] = hw[0];
                slot[1] = hw[1];
            }
            float s = (f[0] + f[1]) + (f[2] + f[3]);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            if ((l16 & 7) == 0) qsum[G * CB + n] = s;
        }
        if (l16 == 0) qsum[NG * CB + n] = ldexpf(1.0f, -e) * p.scale_log2;  // stored after the sums
    }
    __syncthreads();

    const int g = lane >> 2, c = lane & 3;
    float o[NB][A::KS][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < A::KS; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) o[nb][i][j] = 0.0f;
    float m_run[NB][2], l_run[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        m_run[nb][0] = m_run[nb][1] = -INFINITY;
        l_run[nb][0] = l_run[nb][1] = 0.0f;
    }
    // tile t2 of this warp holds stage rows 16 warp + 16 W t2 + {0..15}
    const int r0 = 16 * warp + g, r1 = r0 + 8;
    const int vr[4] = {16 * warp + 2 * c, 16 * warp + 2 * c + 1, 16 * warp + 2 * c + 8, 16 * warp + 2 * c + 9};
    constexpr int TR = 16 * A::W;              // rows between a warp's tiles
    // VLUT 3: the f16 centroid table as byte-permute operands (low bytes of
    // c0..c7, then high bytes); VLUT 2: the four f16 centroids, two per register
    uint32_t tl0 = 0, tl1 = 0, th0 = 0, th1 = 0;
    if constexpr (VLUT == 2) {
        tl0 = (uint32_t)p.cen[0] | ((uint32_t)p.cen[1] << 16);
        tl1 = (uint32_t)p.cen[2] | ((uint32_t)p.cen[3] << 16);
    }
    if constexpr (VLUT == 3)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t cb = p.cen[i], sh = 8 * (i & 3);
            if (i < 4) {
                tl0 |= (cb & 0xFFu) << sh;
                th0 |= (cb >> 8) << sh;
            } else {
                tl1 |= (cb & 0xFFu) << sh;
                th1 |= (cb >> 8) << sh;
            }
        }
    constexpr int QF_NB = gN * A::QCOL;  // bytes of q fragments per block of 8 columns
    const uint32_t qf_lane = smem_addr(qf) + g * A::QCOL + c * 8, lut_a = smem_addr(lut);

    bool ok = true;
    for (int s = 0; s < n_stages; ++s) {
        const int slot = s % p.stages;
        if (!mbar_wait_bounded(full0 + 8 * slot, (s / p.stages) & 1, p.err)) {
            ok = false;
            break;
        }
        const uint32_t kst = smem_addr(stages + slot * p.key_bytes);
        const uint32_t st = smem_addr(stages + p.stages * p.key_bytes + slot * p.stage_bytes);
        const int64_t tile_t0 = t_begin + (int64_t)s * gT + 16 * warp;  // first row of tile 0

        // ---------------- S = Q K^T, group by group, with the group affine, for
        // both tiles; the dequantised key fragments serve every block of columns
        float S[A::TILES][NB][2][2];
#pragma unroll
        for (int t2 = 0; t2 < A::TILES; ++t2)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) S[t2][nb][0][0] = S[t2][nb][0][1] = S[t2][nb][1][0] = S[t2][nb][1][1] = 0.0f;
        // groups two at a time: a row's fp16 scales (zeros) of groups G0, G0 + 1 are
        // one 32-bit word (NG is even, rows are NG * 2 bytes apart)
#pragma unroll 1
        for (int G0 = 0; G0 < A::NG; G0 += 2) {
            uint32_t scp[A::TILES][2], zcp[A::TILES][2];  // [tile][row g, row g + 8]
#pragma unroll
            for (int t2 = 0; t2 < A::TILES; ++t2) {
                const int ra = r0 + TR * t2, rb = r1 + TR * t2;
                scp[t2][0] = g_lds32(st + p.off_ks + (ra * NG + G0) * 2);
                scp[t2][1] = g_lds32(st + p.off_ks + (rb * NG + G0) * 2);
                zcp[t2][0] = g_lds32(st + p.off_kz + (ra * NG + G0) * 2);
                zcp[t2][1] = g_lds32(st + p.off_kz + (rb * NG + G0) * 2);
            }
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
                const int G = G0 + gg;
                uint2 bq[NB][2];
#pragma unroll
                for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) bq[nb][jj] = g_lds64(qf_lane + nb * QF_NB + (2 * G + jj) * 32);
#pragma unroll
                for (int t2 = 0; t2 < A::TILES; ++t2) {
                    const int ra = r0 + TR * t2, rb = r1 + TR * t2;
                    uint32_t k0[4], k1[4];
                    if constexpr (KEY != 0) {
                        key_pairs_sw<D, KEY>(kst, ra, G, c, k0);
                        key_pairs_sw<D, KEY>(kst, rb, G, c, k1);
                    } else {
                        key_pairs<KEY>(kst + ra * p.rbk, G, c, p.kb, k0);
                        key_pairs<KEY>(kst + rb * p.rbk, G, c, p.kb, k1);
                    }
                    const float sc0 = f16_bits_to_f32((uint16_t)(scp[t2][0] >> (16 * gg)));
                    const float sc1 = f16_bits_to_f32((uint16_t)(scp[t2][1] >> (16 * gg)));
                    const float zc0 = f16_bits_to_f32((uint16_t)(zcp[t2][0] >> (16 * gg))) - p.koff;
                    const float zc1 = f16_bits_to_f32((uint16_t)(zcp[t2][1] >> (16 * gg))) - p.koff;
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj)
                            g_mma(acc, k0[2 * jj], k1[2 * jj], k0[2 * jj + 1], k1[2 * jj + 1], bq[nb][jj].x, bq[nb][jj].y);
                        // both columns of the lane at once on packed fp32 pairs
                        const float2 qs = *reinterpret_cast<const float2 *>(&qsum[G * CB + nb * gN + 2 * c]);
                        const float2 s0 = __ffma2_rn(make_float2(sc0, sc0),
                                                     __ffma2_rn(make_float2(zc0, zc0), qs, make_float2(acc[0], acc[1])),
                                                     make_float2(S[t2][nb][0][0], S[t2][nb][0][1]));
                        const float2 s1 = __ffma2_rn(make_float2(sc1, sc1),
                                                     __ffma2_rn(make_float2(zc1, zc1), qs, make_float2(acc[2], acc[3])),
                                                     make_float2(S[t2][nb][1][0], S[t2][nb][1][1]));
                        S[t2][nb][0][0] = s0.x;
                        S[t2][nb][0][1] = s0.y;
                        S[t2][nb][1][0] = s1.x;
                        S[t2][nb][1][1] = s1.y;
                    }
                }
            }
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const float ie0 = qsum[NG * CB + nb * gN + 2 * c], ie1 = qsum[NG * CB + nb * gN + 2 * c + 1];
#pragma unroll
            for (int t2 = 0; t2 < A::TILES; ++t2) {
                S[t2][nb][0][0] *= ie0; S[t2][nb][1][0] *= ie0;
                S[t2][nb][0][1] *= ie1; S[t2][nb][1][1] *= ie1;
            }
        }
        // causal mask: row t is hidden from query row i when t >= base0 + i
        // (this also hides every row past t_end, which is at most the last
        // column's limit, or the split's end when the tile stops there)
#pragma unroll
        for (int t2 = 0; t2 < A::TILES; ++t2) {
            const int64_t tt0 = tile_t0 + TR * t2;
            if (tt0 + 16 > lim_lo) {
                const int64_t ta = tt0 + g - p.base0, tb = ta + 8;
#pragma unroll
                for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int col = col0 + nb * gN + 2 * c + j;
                        const int64_t qi = col < p.cols ? col / p.G : p.M - 1;
                        if (ta >= qi) S[t2][nb][0][j] = -INFINITY;
                        if (tb >= qi) S[t2][nb][1][j] = -INFINITY;
                    }
            }
        }
        // ---------------- online softmax (base 2) over both tiles, columns 2c, 2c+1 of each block
        float pr[A::TILES][NB][2][2];
        bool raise = false;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                raise |= m_run[nb][j] == -INFINITY;
#pragma unroll
                for (int t2 = 0; t2 < A::TILES; ++t2)
                    raise |= S[t2][nb][0][j] > m_run[nb][j] || S[t2][nb][1][j] > m_run[nb][j];
            }
        if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float mt = fmaxf(S[0][nb][0][j], S[0][nb][1][j]);
#pragma unroll
                    for (int t2 = 1; t2 < A::TILES; ++t2) mt = fmaxf(mt, fmaxf(S[t2][nb][0][j], S[t2][nb][1][j]));
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
                    const float mn = fmaxf(m_run[nb][j], mt);
                    const float mu = mn == -INFINITY ? 0.0f : mn;
                    const float alpha = g_ex2(m_run[nb][j] - mu);
                    m_run[nb][j] = mn;
                    float ls = 0.0f;
#pragma unroll
                    for (int t2 = 0; t2 < A::TILES; ++t2) {
                        pr[t2][nb][0][j] = g_ex2(S[t2][nb][0][j] - mu);
                        pr[t2][nb][1][j] = g_ex2(S[t2][nb][1][j] - mu);
                        ls += pr[t2][nb][0][j] + pr[t2][nb][1][j];
                    }
                    l_run[nb][j] = l_run[nb][j] * alpha + ls;
#pragma unroll
                    for (int mt2 = 0; mt2 < A::KS; ++mt2) {
                        o[nb][mt2][j] *= alpha;
                        o[nb][mt2][2 + j] *= alpha;
                    }
                }
        } else {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float ls = 0.0f;
#pragma unroll
                    for (int t2 = 0; t2 < A::TILES; ++t2) {
                        pr[t2][nb][0][j] = g_ex2(S[t2][nb][0][j] - m_run[nb][j]);
                        pr[t2][nb][1][j] = g_ex2(S[t2][nb][1][j] - m_run[nb][j]);
                        ls += pr[t2][nb][0][j] + pr[t2][nb][1][j];
                    }
                    l_run[nb][j] += ls;
                }
        }
        uint32_t pt0[A::TILES][NB], pt1[A::TILES][NB];
        bool vlive[A::TILES][4];
#pragma unroll
        for (int t2 = 0; t2 < A::TILES; ++t2) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                pt0[t2][nb] = g_trans(g_pack_f16x2(pr[t2][nb][0][0], pr[t2][nb][0][1]));  // tokens 2c, 2c+1; column g
                pt1[t2][nb] = g_trans(g_pack_f16x2(pr[t2][nb][1][0], pr[t2][nb][1][1]));  // tokens 2c+8, 2c+9
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) vlive[t2][q] = tile_t0 + TR * t2 + (vr[q] - 16 * warp) < t_end;
        }
        // ---------------- O^T += V^T (P * rms)^T, group by group, both tiles; the
        // value fragments serve every block of columns
        // value scales of groups G, G + 1 (G even) as one 32-bit word per token
        uint32_t svp[A::TILES][4];
#pragma unroll
        for (int G = 0; G < A::NG; ++G) {
            if ((G & 1) == 0)
#pragma unroll
                for (int t2 = 0; t2 < A::TILES; ++t2)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        svp[t2][q] = vlive[t2][q] ? g_lds32(st + p.off_vs + ((vr[q] + TR * t2) * NG + G) * 2) : 0u;
#pragma unroll
            for (int t2 = 0; t2 < A::TILES; ++t2) {
                // the two tokens' scales of group G as one f16 pair
                const uint32_t sel = (G & 1) ? 0x7632u : 0x5410u;
                const uint32_t sv01 = __byte_perm(svp[t2][0], svp[t2][1], sel), sv23 = __byte_perm(svp[t2][2], svp[t2][3], sel);
                // a[half]: rows g, g+8 of the m-tile = dims 32G + 4g + 2 half + {0, 1};
                // registers 0, 1 pair tokens q0, q1, registers 2, 3 tokens q2, q3
                uint32_t a[2][4];
                if constexpr (VLUT == 2) {
                    // the four tokens' 8-bit fields (dims 32G + 4g .. +3) are bytes; per
                    // dim r and token pair, selector nibbles (2a, 2a+1, 2b, 2b+1) pick the
                    // f16 centroids c[a], c[b] of the two tokens' codes in one permute
                    uint32_t x[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) x[q] = g_lds8(st + p.off_v + (vr[q] + TR * t2) * p.rbv + 8 * G + g);
#pragma unroll
                    for (int pr2 = 0; pr2 < 2; ++pr2) {
                        const uint32_t u = x[2 * pr2] | (x[2 * pr2 + 1] << 8);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint32_t ab = (u >> (2 * r)) & 0x0303u;  // code of the first token, of the second
                            a[r >> 1][2 * pr2 + (r & 1)] = __byte_perm(tl0, tl1, ab * 0x22u + 0x1010u);
                        }
                    }
                } else if constexpr (VLUT == 3) {
                    // the four tokens' 12-bit fields (dims 32G + 4g .. +3), two tokens side
                    // by side, spread to one code per nibble, looked up 4 at a time
                    const int bit = (32 * G + 4 * g) * 3;
                    uint32_t x[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t ad = st + p.off_v + (vr[q] + TR * t2) * p.rbv + 4 * (bit >> 5);
                        x[q] = __funnelshift_r(g_lds32(ad), g_lds32(ad + 4), bit & 31);
                    }
#pragma unroll
                    for (int pr2 = 0; pr2 < 2; ++pr2) {
                        const uint32_t w = __byte_perm(x[2 * pr2], x[2 * pr2 + 1], 0x5410u);
                        const uint32_t y = (w & 0x003F003Fu) | ((w & 0x0FC00FC0u) * 4u);
                        // each byte of y holds two codes; adding the upper one to itself
                        // moves it to bits 4-6, and nothing carries out of a byte
                        const uint32_t e = y + (y & 0x38383838u);
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const uint32_t sel = __byte_perm(e, 0u, half ? 0x0031u : 0x0020u);
                            const uint32_t lo = __byte_perm(tl0, tl1, sel), hi = __byte_perm(th0, th1, sel);
                            a[half][2 * pr2] = __byte_perm(lo, hi, 0x6240u);      // dim r: (first, second)
                            a[half][2 * pr2 + 1] = __byte_perm(lo, hi, 0x7351u);  // dim r + 1
                        }
                    }
                } else {
                    uint32_t hv[4][4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) value_quad(st + p.off_v + (vr[q] + TR * t2) * p.rbv, G, g, p.vb, lut_a, hv[q]);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int r = 2 * half;
                        a[half][0] = hv[0][r] | (hv[1][r] << 16);
                        a[half][1] = hv[0][r + 1] | (hv[1][r + 1] << 16);
                        a[half][2] = hv[2][r] | (hv[3][r] << 16);
                        a[half][3] = hv[2][r + 1] | (hv[3][r + 1] << 16);
                    }
                }
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    const uint32_t b0 = g_hmul2(pt0[t2][nb], sv01), b1 = g_hmul2(pt1[t2][nb], sv23);
#pragma unroll
                    for (int half = 0; half < 2; ++half)
                        g_mma(o[nb][2 * G + half], a[half][0], a[half][1], a[half][2], a[half][3], b0, b1);
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&done[slot], 1u) == A::W - 1) {
                done[slot] = 0;
                if (s + p.stages < n_stages) issue(s + p.stages);
            }
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- merge the warps
    float *mw = merge + warp * CB * (D + 2);  // [column][D] o, then [column] m, [column] l
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            l_run[nb][j] += __shfl_xor_sync(0xffffffffu, l_run[nb][j], 4);
            l_run[nb][j] += __shfl_xor_sync(0xffffffffu, l_run[nb][j], 8);
            l_run[nb][j] += __shfl_xor_sync(0xffffffffu, l_run[nb][j], 16);
        }
#pragma unroll
        for (int mt = 0; mt < A::KS; ++mt) {
            const int G = mt >> 1, half = mt & 1;
            const int d0 = 32 * G + 4 * g + 2 * half;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mw[(nb * gN + 2 * c + j) * D + d0] = o[nb][mt][j];
                mw[(nb * gN + 2 * c + j) * D + d0 + 1] = o[nb][mt][2 + j];
            }
        }
        if (g == 0) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mw[CB * D + nb * gN + 2 * c + j] = ok ? m_run[nb][j] : -INFINITY;
                mw[CB * D + CB + nb * gN + 2 * c + j] = ok ? l_run[nb][j] : 0.0f;
            }
        }
    }
    __syncthreads();
    // thread -> (column hh, a D/16 slice of dims), one block of 8 columns at a time
    constexpr int PER = D / 16;
    const int d0 = (threadIdx.x & 15) * PER;
#pragma unroll 1
    for (int hh = threadIdx.x >> 4; hh < CB; hh += A::THREADS / 16) {
        float mmax = -INFINITY;
#pragma unroll
        for (int w = 0; w < A::W; ++w) mmax = fmaxf(mmax, merge[w * CB * (D + 2) + CB * D + hh]);
        const float mu = mmax == -INFINITY ? 0.0f : mmax;
        float ov[PER], lsum = 0.0f;
#pragma unroll
        for (int i = 0; i < PER; ++i) ov[i] = 0.0f;
#pragma unroll
        for (int w = 0; w < A::W; ++w) {
            const float *m2 = merge + w * CB * (D + 2);
            const float wt = g_ex2(m2[CB * D + hh] - mu);
            lsum += m2[CB * D + CB + hh] * wt;
#pragma unroll
            for (int i = 0; i < PER; ++i) ov[i] += m2[hh * D + d0 + i] * wt;
        }
        const int64_t pidx = ((bh * p.HB + hb) * p.splits + split) * CB + hh;
        float4 *dst = reinterpret_cast<float4 *>(p.part_o + pidx * D + d0);
#pragma unroll
        for (int i = 0; i < PER / 4; ++i) dst[i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
        if ((threadIdx.x & 15) == 0) {
            p.part_ml[2 * pidx] = mmax;
            p.part_ml[2 * pidx + 1] = lsum;
        }
    }
}

// ---------------------------------------------------------------- combine + deferred un-rotation
struct GenCombineParams {
    const float *part_o, *part_ml;
    float *out;  // [B][M][QH][D]
    int H, QH, G, M, HB, CB, splits, rows;
    float inv_sqrt_d;
    SignBits sg;  // value signs
};

// Each (sequence, query row, q-head) row takes W warps (1, 4, 16 or 32 as the
// splits grow); a CTA holds max(4, W) warps.  Lane holds dims PER*lane ..
// +PER-1.  Warp w of a row merges the splits w, w + W, ...: up to gFew<D>()
// of them with every load issued before any is used (one memory round trip),
// more in chunks of 32 whose (max, sum) pairs are read one per lane, the
// weights broadcast and the chunk's output rows read with independent loads.
// The row's first warp then merges its warps' results.
constexpr int gCombineWarps = 4;
template <int D>
__host__ __device__ constexpr int gFew() { return 32 / (D / 32) > 2 ? 32 / (D / 32) : 2; }
__host__ __device__ constexpr int g_combine_cta_warps(int W) { return W > gCombineWarps ? W : gCombineWarps; }

template <int D, int W>
__global__ void __launch_bounds__(g_combine_cta_warps(W) * 32) attn_generic_combine(const __grid_constant__ GenCombineParams p)
{
    constexpr int PER = D / 32, CW = g_combine_cta_warps(W), KF = gFew<D>();
    __shared__ float wo[W > 1 ? CW : 1][PER][32];  // [warp][k][lane]: conflict-free
    __shared__ float wm[CW], wl[CW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * (CW / W) + warp / W, wid = warp % W, lead = warp - wid;
    const bool live = row < p.rows;
    pdl_wait_primary();  // the partials' writer has completed and its writes are visible
    pdl_allow_dependents();
    if (W == 1 && !live) return;  // no barrier below when W = 1
    const int per_seq = p.M * p.QH;
    const int b = row / per_seq, rem = row - b * per_seq, i = rem / p.QH, qh = rem - i * p.QH;
    const int h = qh / p.G, col = i * p.G + (qh - h * p.G), hb = col / p.CB, n = col - hb * p.CB;
    const int64_t base = (((int64_t)b * p.H + h) * p.HB + hb) * p.splits;
    const int n_mine = live && p.splits > wid ? (p.splits - wid + W - 1) / W : 0;
    auto split_index = [&](int j) { return (base + wid + (int64_t)W * j) * p.CB + n; };
    float mw = -INFINITY;
    float x[PER], l = 0.0f;
#pragma unroll
    for (int k = 0; k < PER; ++k) x[k] = 0.0f;
    if (n_mine <= KF) {
        float2 ml = make_float2(-INFINITY, 0.0f);
        if (lane < n_mine) ml = *reinterpret_cast<const float2 *>(p.part_ml + 2 * split_index(lane));
        float v[KF][PER];
#pragma unroll
        for (int j = 0; j < KF; ++j) {
            const float *src = p.part_o + split_index(j) * D + PER * lane;
#pragma unroll
            for (int k = 0; k < PER; ++k) v[j][k] = j < n_mine ? src[k] : 0.0f;
        }
        mw = ml.x;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
        const float muw = mw == -INFINITY ? 0.0f : mw;
        const float wt = lane < n_mine ? g_ex2(ml.x - muw) : 0.0f;
        if (lane < n_mine) l = ml.y * wt;
#pragma unroll
        for (int j = 0; j < KF; ++j) {
            const float w = __shfl_sync(0xffffffffu, wt, j);
#pragma unroll
            for (int k = 0; k < PER; ++k) x[k] += v[j][k] * w;
        }
    } else {
        for (int j = lane; j < n_mine; j += 32) mw = fmaxf(mw, p.part_ml[2 * split_index(j)]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
        const float muw = mw == -INFINITY ? 0.0f : mw;
        for (int i0 = 0; i0 < n_mine; i0 += 32) {
            float wt = 0.0f;
            if (i0 + lane < n_mine) {
                const float2 ml = *reinterpret_cast<const float2 *>(p.part_ml + 2 * split_index(i0 + lane));
                wt = g_ex2(ml.x - muw);
                l += ml.y * wt;
            }
            const int cnt = n_mine - i0 < 32 ? n_mine - i0 : 32;
#pragma unroll 4
            for (int j = 0; j < cnt; ++j) {
                const float w = __shfl_sync(0xffffffffu, wt, j);
                const float *src = p.part_o + split_index(i0 + j) * D + PER * lane;
#pragma unroll
                for (int k = 0; k < PER; ++k) x[k] += src[k] * w;
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if constexpr (W > 1) {
#pragma unroll
        for (int k = 0; k < PER; ++k) wo[warp][k][lane] = x[k];
        if (lane == 0) {
            wm[warp] = mw;
            wl[warp] = l;
        }
        __syncthreads();
        if (wid != 0 || !live) return;
        float mmax = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) mmax = fmaxf(mmax, wm[lead + w]);
        const float mu = mmax == -INFINITY ? 0.0f : mmax;
        l = 0.0f;
#pragma unroll
        for (int k = 0; k < PER; ++k) x[k] = 0.0f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            // a warp without live splits carries zeros; the others rescale to the common max
            const float wt = wm[lead + w] == -INFINITY ? 0.0f : g_ex2(wm[lead + w] - mu);
            l += wl[lead + w] * wt;
#pragma unroll
            for (int k = 0; k < PER; ++k) x[k] += wo[lead + w][k][lane] * wt;
        }
    }
    const float inv_l = 1.0f / l;
#pragma unroll
    for (int k = 0; k < PER; ++k) x[k] *= inv_l;
    // inverse transform in Sylvester order: log2(PER) stages in-lane, 5 across lanes
#pragma unroll
    for (int hs = 1; hs < PER; hs <<= 1)
#pragma unroll
        for (int k = 0; k < PER; k += 2 * hs)
#pragma unroll
            for (int j = k; j < k + hs; ++j) {
                const float a = x[j], bb = x[j + hs];
                x[j] = a + bb;
                x[j + hs] = a - bb;
            }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const float other = __shfl_xor_sync(0xffffffffu, x[k], m);
            x[k] = upper ? other - x[k] : x[k] + other;
        }
    }
    float *dst = p.out + (int64_t)row * D + PER * lane;
#pragma unroll
    for (int k = 0; k < PER; ++k) dst[k] = x[k] * (sign_negative(p.sg, PER * lane + k) ? -p.inv_sqrt_d : p.inv_sqrt_d);
}

// ---------------------------------------------------------------- host side
// The fewest warps per row (1, 4, 16, 32; 16 at most at head_dim 512, whose
// partials of 32 warps would not fit static shared memory) that give each
// warp at most gFew<D>() splits; one warp per row packs 4 rows per CTA.  The
// merge is a programmatic dependent of the kernel that wrote the partials (it
// waits for that grid before reading them).
template <int D>
cudaError_t launch_generic_combine(const GenCombineParams &cp, cudaStream_t s)
{
    constexpr int KF = gFew<D>();
    if (cp.splits <= KF)
        return launch_dependent(attn_generic_combine<D, 1>, dim3((cp.rows + gCombineWarps - 1) / gCombineWarps),
                                dim3(gCombineWarps * 32), 0, s, cp);
    if (cp.splits <= 4 * KF) return launch_dependent(attn_generic_combine<D, 4>, dim3(cp.rows), dim3(4 * 32), 0, s, cp);
    if (D == 512 || cp.splits <= 16 * KF)
        return launch_dependent(attn_generic_combine<D, 16>, dim3(cp.rows), dim3(16 * 32), 0, s, cp);
    if constexpr (D < 512) return launch_dependent(attn_generic_combine<D, 32>, dim3(cp.rows), dim3(32 * 32), 0, s, cp);
    return cudaErrorInvalidValue;
}

struct GenPlan {
    int nb, hb, splits, stages, stage_bytes, smem;
    int vlut;  // VLUT of the instantiation: 3 or 2 for 3- or 2-bit values, else 0
    int key;   // KEY of the instantiation: 8 or 4 for 8- or 4-bit keys, else 0
    int64_t tokens_per_split;
    int off_ks, off_kz, off_vs, off_v, key_bytes;
};

// blocks of 8 columns per CTA: enough to cover the columns of one kv-head in
// a single pass over its cache rows, capped by the accumulator registers
inline int gen_nb(int d, int64_t cols)
{
    const int cap = d <= 128 ? 4 : (d == 256 ? 2 : 1);
    const int64_t need = (cols + gN - 1) / gN;
    const int nb = need <= 1 ? 1 : (need <= 2 ? 2 : 4);
    return nb < cap ? nb : cap;
}

// Calls f with the kernel instantiation the plan's VLUT and KEY name.
template <int D, int NB, int VLUT, typename F>
auto gen_dispatch_key(const GenPlan &pl, F &&f)
{
    return pl.key == 8 ? f(attn_generic_kernel<D, NB, VLUT, 8>)
           : pl.key == 4 ? f(attn_generic_kernel<D, NB, VLUT, 4>)
                         : f(attn_generic_kernel<D, NB, VLUT, 0>);
}

template <int D, int NB, typename F>
auto gen_dispatch(const GenPlan &pl, F &&f)
{
    return pl.vlut == 3   ? gen_dispatch_key<D, NB, 3>(pl, f)
           : pl.vlut == 2 ? gen_dispatch_key<D, NB, 2>(pl, f)
                          : gen_dispatch_key<D, NB, 0>(pl, f);
}

template <int D, int NB>
bool gen_plan_nb(const CacheView &c, int q_heads, int64_t m, int64_t seq_len, GenPlan &pl)
{
    using A = GGeo<D, NB>;
    const int NG = D / 32, rbk = D * c.kb / 8, rbv = D * c.vb / 8;
    auto r16 = [](int x) { return (x + 15) / 16 * 16; };
    pl.nb = NB;
    pl.vlut = c.vb == 3 ? 3 : (c.vb == 2 ? 2 : 0);
    // 8- and 4-bit keys take swizzled tensor copies (row coordinates are 32-bit)
    pl.key = (int64_t)c.B * c.H * c.cap < (int64_t(1) << 31) ? (c.kb == 8 ? 8 : (c.kb == 4 ? 4 : 0)) : 0;
    pl.key_bytes = pl.key != 0 ? (gT * rbk + 1023) / 1024 * 1024 : r16(gT * rbk);
    pl.off_ks = 0;
    pl.off_kz = pl.off_ks + r16(gT * NG * 2);
    pl.off_vs = pl.off_kz + r16(gT * NG * 2);
    pl.off_v = pl.off_vs + r16(gT * NG * 2);
    pl.stage_bytes = r16(pl.off_v + gT * rbv + 16);
    pl.stages = 2;  // with 2-warp CTAs a deeper ring only costs resident CTAs
    const int ring = pl.stages * (pl.key_bytes + pl.stage_bytes) > A::MERGE ? pl.stages * (pl.key_bytes + pl.stage_bytes)
                                                                           : A::MERGE;
    pl.smem = 1024 /*align slack*/ + ring + A::QF + A::QS + (pl.vlut == 0 ? 512 : 0) /*lut*/ +
              gMaxStages * 12 /*barriers, counters*/;
    const int per_sm = gen_dispatch<D, NB>(pl, [&](auto kern) {
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem) != cudaSuccess) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, GGeo<D, NB>::THREADS, pl.smem) != cudaSuccess)
            return 0;
        return n;
    });
    if (per_sm < 1) return false;
    const int64_t cols = (int64_t)(q_heads / c.H) * m;
    pl.hb = (int)((cols + A::CB - 1) / A::CB);
    const int64_t units = (int64_t)c.B * c.H * pl.hb;
    const int64_t nst = (seq_len + gT - 1) / gT;
    const int64_t slots = (int64_t)num_sms() * per_sm;
    pl.splits = 1;
    pl.tokens_per_split = nst * gT;
    double best = 1e300;
    for (int waves = 1; waves <= 16; ++waves) {
        int64_t s = (waves * slots + units - 1) / units;
        if (s < 1) s = 1;
        if (s > nst) s = nst;
        const int64_t per = (nst + s - 1) / s, sp = (nst + per - 1) / per;
        const double cost = (double)((units * sp + slots - 1) / slots) * (double)(per + 2);
        if (cost < best - 1e-9) {
            best = cost;
            pl.splits = (int)sp;
            pl.tokens_per_split = per * gT;
        }
    }
    return true;
}

template <int D>
bool gen_plan(const CacheView &c, int q_heads, int64_t m, int64_t seq_len, GenPlan &pl)
{
    switch (gen_nb(D, (int64_t)(q_heads / c.H) * m)) {
    case 1: return gen_plan_nb<D, 1>(c, q_heads, m, seq_len, pl);
    case 2: if constexpr (D <= 256) return gen_plan_nb<D, 2>(c, q_heads, m, seq_len, pl); break;
    case 4: if constexpr (D <= 128) return gen_plan_nb<D, 4>(c, q_heads, m, seq_len, pl); break;
    }
    return false;
}

template <int D, int NB>
cudaError_t gen_launch(const GenPlan &pl, dim3 grid, const CUtensorMap &kmap, const GenParams &p, cudaStream_t s)
{
    return gen_dispatch<D, NB>(
        pl, [&](auto kern) { return launch_dependent(kern, grid, dim3(GGeo<D, NB>::THREADS), (size_t)pl.smem, s, kmap, p); });
}

// Tensor map over the key plane for the swizzled key tiles of 8- and 4-bit
// keys: [B H cap rows][row bytes], boxes of BOXB bytes x gT rows.
template <int D>
bool gen_key_map(const CacheView &c, CUtensorMap *map)
{
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const int rb = D * c.kb / 8, boxb = rb < 128 ? rb : 128;
    const cuuint64_t gdim[2] = {(cuuint64_t)rb, (cuuint64_t)c.B * c.H * c.cap};
    const cuuint64_t gstride[1] = {(cuuint64_t)rb};
    const cuuint32_t box[2] = {(cuuint32_t)boxb, (cuuint32_t)gT};
    const cuuint32_t estride[2] = {1, 1};
    const CUtensorMapSwizzle sw = boxb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : boxb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c.k_codes, gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
              sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
size_t gen_workspace(const CacheView &c, int q_heads, int64_t m, int64_t seq_len)
{
    GenPlan pl;
    if (!gen_plan<D>(c, q_heads, m, seq_len, pl)) return 0;
    return (size_t)c.B * c.H * pl.hb * pl.splits * gN * pl.nb * (D + 2) * 4;
}

template <int D>
cudaError_t gen_run(const CacheView &c, const uint16_t *q, int QH, int64_t m, int64_t seq_len, float scale, float *out,
                    void *ws, size_t ws_bytes, cudaStream_t s)
{
    GenPlan pl;
    if (!gen_plan<D>(c, QH, m, seq_len, pl)) return cudaErrorInvalidConfiguration;
    const int G = QH / c.H, CB = gN * pl.nb;
    const size_t parts = (size_t)c.B * c.H * pl.hb * pl.splits * CB;
    const size_t need_o = parts * D * 4;
    if (ws_bytes < need_o + parts * 2 * 4) return cudaErrorInvalidValue;
    GenParams p{};
    p.k_codes = c.k_codes;
    p.v_codes = c.v_codes;
    p.k_scale = c.k_scale;
    p.k_zero = c.k_zero;
    p.v_scale = c.v_scale;
    p.q = q;
    p.part_o = static_cast<float *>(ws);
    p.part_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + need_o);
    p.err = device_error_word();
    if (!p.err) return cudaErrorInvalidDevice;
    p.H = c.H;
    p.QH = QH;
    p.G = G;
    p.M = (int)m;
    p.cols = G * (int)m;
    p.HB = pl.hb;
    p.splits = pl.splits;
    p.kb = c.kb;
    p.vb = c.vb;
    p.stages = pl.stages;
    p.cap = c.cap;
    p.seq_len = seq_len;
    p.tokens_per_split = pl.tokens_per_split;
    p.base0 = seq_len - m + 1;
    p.rbk = D * c.kb / 8;
    p.rbv = D * c.vb / 8;
    p.off_ks = pl.off_ks;
    p.off_kz = pl.off_kz;
    p.off_vs = pl.off_vs;
    p.off_v = pl.off_v;
    p.stage_bytes = pl.stage_bytes;
    p.key_bytes = pl.key_bytes;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.koff = c.kb == 8 ? 1152.0f : 1024.0f;
    const Tables &tab = codebook_tables(c.vb);
    for (int i = 0; i < (1 << c.vb); ++i) p.cen[i] = __half_as_ushort(__float2half_rn(tab.centroids[i]));
    if ((int64_t)c.H * pl.hb > 65535 || c.B > 65535) return cudaErrorInvalidValue;
    CUtensorMap kmap{};
    if (pl.key != 0 && !gen_key_map<D>(c, &kmap)) return cudaErrorInvalidValue;
    const dim3 grid(pl.splits, c.H * pl.hb, c.B);
    cudaError_t e = cudaErrorInvalidValue;
    switch (pl.nb) {
    case 1: e = gen_launch<D, 1>(pl, grid, kmap, p, s); break;
    case 2: if constexpr (D <= 256) e = gen_launch<D, 2>(pl, grid, kmap, p, s); break;
    case 4: if constexpr (D <= 128) e = gen_launch<D, 4>(pl, grid, kmap, p, s); break;
    }
    if (e != cudaSuccess) return e;
    const int rows = c.B * (int)m * QH;
    GenCombineParams cp{p.part_o, p.part_ml, out, c.H, QH, G, (int)m, pl.hb, CB, pl.splits, rows,
                        inv_sqrt_head_dim(D), c.signs};
    return launch_generic_combine<D>(cp, s);
}

template <int D>
cudaError_t combine_parts(const float *part_o, const float *part_ml, float *out, int B, int H, int QH, int m, int hb,
                          int cb, int splits, const SignBits &sg, cudaStream_t s)
{
    const int rows = B * m * QH;
    GenCombineParams cp{part_o, part_ml, out, H, QH, QH / H, m, hb, cb, splits, rows, inv_sqrt_head_dim(D), sg};
    return launch_generic_combine<D>(cp, s);
}

}  // namespace
}  // namespace tq

// The entry points of one head_dim's translation unit.
#define TQ_ATTENTION_GENERIC_ENTRIES(D)                                                                                  \
    namespace tq {                                                                                                       \
    cudaError_t launch_attention_generic_d##D(const CacheView &c, const uint16_t *q, int q_heads, int64_t m,            \
                                              int64_t seq_len, float scale, float *out, void *ws, size_t ws_bytes,     \
                                              cudaStream_t s)                                                          \
    {                                                                                                                    \
        return gen_run<D>(c, q, q_heads, m, seq_len, scale, out, ws, ws_bytes, s);                                       \
    }                                                                                                                    \
    size_t attention_generic_workspace_d##D(const CacheView &c, int q_heads, int64_t m, int64_t seq_len)               \
    {                                                                                                                    \
        return gen_workspace<D>(c, q_heads, m, seq_len);                                                                 \
    }                                                                                                                    \
    cudaError_t launch_attention_combine_parts_d##D(const float *part_o, const float *part_ml, float *out, int B,      \
                                                    int H, int QH, int m, int hb, int cb, int splits,                  \
                                                    const SignBits &sg, cudaStream_t s)                                \
    {                                                                                                                    \
        return combine_parts<D>(part_o, part_ml, out, B, H, QH, m, hb, cb, splits, sg, s);                               \
    }                                                                                                                    \
    }
