// tq_attention.cu -- fused dequantise-on-fetch GQA decode attention.
//
// Method: mlx-bun "TurboQuant -- rotation-based quantization", Part A:
// "Architecture in mlx-bun" (dequantize-on-fetch: attention reads the
// dequantised window; the token being generated is appended first), the
// "Algorithm" section (key and value dequantisation), and "Deferred inverse
// FWHT" (attention is linear in V, so the weighted sum is formed in the
// rotated domain and un-rotated once per query row).  GQA replicates whole
// kv-heads: q-head h reads kv-head h / G.
//
// GB300 design (one GPU, sm_103a), for head_dims 64, 128 and 256 with 8- or
// 4-bit keys and 2-, 3- or 4-bit values:
//  * Split-KV: CTA (split, kv-head, sequence) streams its token range through
//    a 2-stage shared-memory ring; each of its 2 warps takes two 16-token tiles
//    of a 64-token stage (four of a 128-token stage at head_dim 64, whose rows
//    are short; three of a 96-token stage at head_dim 128 with 4-bit keys) and
//    works on them at once (independent dependency chains to interleave).  A
//    stage is 2-D TMA loads of the key codes (boxes of at most 128 bytes per
//    row -- two at head_dim 256 with 8-bit keys -- with the swizzle of the box
//    width, so the per-row fragment reads of the MMA are bank-conflict-free)
//    and four 1-D bulk copies of the other planes, completing on the slot's
//    mbarrier; the last warp to finish a stage issues the copies that refill
//    its slot, so no warp is set aside as a producer (8 CTAs fit on an SM at
//    head_dims 64 and 128, 4 at 256).
//  * QK^T on tensor cores (mma.sync m16n8k16, f16 in, f32 accumulate): M = 16
//    tokens, N = 8 columns: 8 of the G q-heads sharing the kv-head, K =
//    head_dim.  A group above 8 has ceil(G/8) column blocks: at head_dims 64
//    and 128 a CTA takes two of them, so the key and value codes it unpacks
//    serve 16 columns (4 CTAs per SM at 128, for the doubled registers); at
//    256 each block is its own CTA, neighbours in the grid so their reads of
//    the same rows meet in L2.  Columns past G repeat the last head and are
//    dropped.  Key codes become exact f16 integers with one logic op each:
//    offset + code (a shift first for the upper bytes; 4-bit codes in odd
//    nibbles are read in place as 1024 + 16 code, their q taken / 16), so
//    S = sum_g scale_g * (acc_g + zero_g * sum_{j in g} q_j - offsets' share)
//    -- the per-group affine is applied to the 8-head scores, not to each
//    element.
//  * PV in the rotated domain (mma.sync, M = 16 dims, N = 8 heads, K = 16
//    tokens): value codes are mapped to f16 centroids by byte-permute table
//    lookups in registers (3 bits: four codes spread to nibbles per lookup;
//    2 bits: one f16 pair of the four centroids per lookup; 4 bits: the
//    magnitude index and sign of each code, the table being odd); the
//    per-group RMS scale is folded into P.
//  * Online softmax (base 2) per warp; warps merge in shared memory; each CTA
//    writes (max, sum, unnormalised o) per head.  A second kernel merges the
//    splits (log-sum-exp) and applies the inverse transform and signs once per
//    (sequence, q-head): the one below at head_dim 128, the generic kernel's
//    (same partial layout) at 64 and 256.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tq_common.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kG = 8;              // MMA columns: a block of 8 of a kv-head's q-heads
constexpr int kCW = 2;             // warps per CTA (all compute; the last to finish a stage refills it)
constexpr int kThreads = kCW * 32;
constexpr int kStages = 2;         // ring depth (8 CTAs of 2 x 13 KB fit on an SM)
constexpr float kOffset8 = 1152.0f;  // 8-bit keys: f16 value = 1152 + signed code

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

// blocks of kG q-heads (MMA columns) per kv-head
inline int col_blocks(int group) { return (group + kG - 1) / kG; }

// NBC: column blocks per CTA (2 at head_dims up to 128 when a kv-head has
// more than kG q-heads: the key and value codes are unpacked once for both)
template <int KB, int D, int VB, int NBC = 1>
struct AGeo {
    // 16-token tiles per warp and stage, worked on together, and tokens per
    // stage: with one column block, four at head_dim 64 and three at 128 with
    // 4-bit keys (short rows: the per-stage work is spread over more of them;
    // the registers and the 2-slot ring still fit 8 CTAs on an SM)
    static constexpr int TILES = NBC != 1 ? 2 : D == 64 ? 4 : (D == 128 && KB == 4) ? 3 : 2;
    static constexpr int ST = 16 * TILES * kCW;
    static constexpr int NG = D / 32;                          // groups per row
    static constexpr int KROW = D * KB / 8;                    // key code bytes per token
    static constexpr int SW = KROW < 128 ? KROW : 128;         // key box row bytes = swizzle span
    static constexpr int NBOX = KROW / SW;                     // key boxes per row
    static constexpr int RBV = D * VB / 8;                     // value code bytes per token
    static constexpr int K_BYTES = ST * KROW;
    static constexpr int SC_BYTES = ST * NG * 2;               // one fp16 plane
    static constexpr int V_BYTES = ST * RBV;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_KS = K_BYTES;
    static constexpr int OFF_KZ = OFF_KS + SC_BYTES;
    static constexpr int OFF_VS = OFF_KZ + SC_BYTES;
    static constexpr int OFF_V = OFF_VS + SC_BYTES;
    static constexpr int STAGE = round_up(OFF_V + V_BYTES + 16, 1024);  // 1024: swizzle atom alignment
    static constexpr int MERGE = kCW * NBC * kG * (D + 2) * 4;        // per-warp partials (reuse the ring)
    static constexpr int RING = kStages * STAGE > MERGE ? kStages * STAGE : MERGE;
    static constexpr int SMEM = 1024 /*align slack*/ + RING + kStages * 8 /*full barriers*/ + kStages * 4 /*counters*/;
    // resident CTAs per SM the register budget is sized for (head_dim 256, or
    // two column blocks, hold twice the q fragments and output accumulators)
    static constexpr int MIN_BLOCKS = D * NBC >= 256 ? 4 : 8;
};

struct AttnParams {
    const uint16_t *k_scale, *k_zero, *v_scale;
    const uint8_t *v_codes;
    const uint16_t *q;  // [B][QH][D] bf16
    float *part_o;      // [B][H][S][G][D]
    float *part_ml;     // [B][H][S][G][2]
    int H, QH, G, NB, splits;  // G = QH / H q-heads per kv-head; NB = ceil(G / kG) column blocks
    int64_t cap, seq_len, tokens_per_split;
    float scale_log2;  // softmax_scale * log2(e)
    uint32_t *err;
    // value centroids as byte-permute tables: 3 bits -- low bytes of the f16
    // c0..c7 (tl0, tl1), then their high bytes (th0, th1); 2 bits -- the f16
    // c0, c1 (tl0) and c2, c3 (tl1); 4 bits -- low and high bytes of the f16
    // magnitudes c8..c15 (the table is odd: c[15 - k] = -c[k])
    uint32_t tl0, tl1, th0, th1;
    uint32_t k_const, k_flip;     // key byte -> f16 (1024 + byte ^ 0x80) as one logic op (see below)
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint2 lds64(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// N consecutive 32-bit words of shared memory (N = 1, 2 or 4; the address aligned to 4 N bytes)
template <int N>
__device__ __forceinline__ void lds_words(uint32_t a, uint32_t (&w)[N])
{
    if constexpr (N == 1) {
        w[0] = lds32(a);
    } else if constexpr (N == 2) {
        const uint2 v = lds64(a);
        w[0] = v.x;
        w[1] = v.y;
    } else {
        static_assert(N == 4, "one, two or four words");
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(a));
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Byte permute, default mode (used as an 8-entry table lookup: each selector
// nibble 0..7 picks one byte of the table held in a and b).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Key codes -> a pair of exact f16 integers in one 3-input logic op: where
// k_const has a bit set the result takes k_flip's bit (the f16 exponent
// pattern of 1024), elsewhere the code bit xor k_flip's bit (0x80 turns an
// int8 code into offset binary).  The f16 value is 1024 + (offset) code.
__device__ __forceinline__ uint32_t kcvt(uint32_t w, const AttnParams &p)
{
    return (p.k_const & p.k_flip) | (~p.k_const & (w ^ p.k_flip));
}

// Right shift done on the multiply-add pipe (the integer/logic pipe is the
// bottleneck of this kernel): x >> k == high word of x * 2^(32-k).
template <int K>
__device__ __forceinline__ uint32_t shr_fma(uint32_t x)
{
    return __umulhi(x, 1u << (32 - K));
}

// ---------------------------------------------------------------- the split kernel
template <int KB, int D, int VB, int NBC>
__global__ void __launch_bounds__(kThreads, AGeo<KB, D, VB, NBC>::MIN_BLOCKS)
    attn_split_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ AttnParams p)
{
    using A = AGeo<KB, D, VB, NBC>;
    constexpr int NG = A::NG;
    constexpr int NH = NBC * kG;  // MMA columns of the CTA
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    float *merge = reinterpret_cast<float *>(smem);  // after the loop, reuses the ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + A::RING);
    uint32_t *done = reinterpret_cast<uint32_t *>(smem + A::RING + kStages * 8);
    const uint32_t full0 = smem_addr(bars);

    pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // blockIdx.y = (kv-head, NBC blocks of kG q-heads); the CTAs of one kv-head
    // are neighbours in the grid, so their reads of the same rows meet in L2
    const int nbp = (p.NB + NBC - 1) / NBC;  // CTAs per kv-head
    const int split = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    const int h = hv / nbp, hb0 = (hv - h * nbp) * NBC;  // the CTA's first column block
    const int64_t bh = (int64_t)b * p.H + h;
    const int64_t t_begin = (int64_t)split * p.tokens_per_split;
    const int64_t t_end = imin64(p.seq_len, t_begin + p.tokens_per_split);
    const int n_stages = t_end > t_begin ? (int)((t_end - t_begin + A::ST - 1) / A::ST) : 0;

    // stage s -> ring slot s % kStages: one 2-D TMA load (key codes) and four
    // 1-D bulk copies (the other planes) completing on the slot's barrier
    auto issue = [&](int s) {
        const int slot = s % kStages;
        const int64_t t = t_begin + (int64_t)s * A::ST;
        const int rows = (int)imin64(A::ST, p.cap - t);  // multiple of 16
        const int64_t row0 = bh * p.cap + t;
        const uint32_t st = smem_addr(stages + slot * A::STAGE), bar = full0 + 8 * slot;
        mbar_arrive_expect_tx(bar, (uint32_t)(A::K_BYTES + rows * (3 * NG * 2 + A::RBV)));
#pragma unroll
        for (int j = 0; j < A::NBOX; ++j)  // key rows wider than 128 bytes arrive as several boxes
            tma_load_2d(st + A::OFF_K + j * (A::ST * A::SW), &kmap, j * A::SW, (int)row0, bar);
        bulk_g2s(st + A::OFF_KS, p.k_scale + row0 * NG, rows * NG * 2, bar);
        bulk_g2s(st + A::OFF_KZ, p.k_zero + row0 * NG, rows * NG * 2, bar);
        bulk_g2s(st + A::OFF_VS, p.v_scale + row0 * NG, rows * NG * 2, bar);
        bulk_g2s(st + A::OFF_V, p.v_codes + row0 * A::RBV, rows * A::RBV, bar);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            done[s] = 0;
        }
        fence_mbar_init();
        for (int s = 0; s < kStages && s < n_stages; ++s) issue(s);
    }
    __syncthreads();

    // ---------------------------------------------------------------- compute warps
    const int g = lane >> 2, c = lane & 3;
    // Q fragments (B operand of QK^T): head n = g; per k-step two f16x2 registers.
    // The dim order inside a 32-group is permuted to match how key codes unpack.
    uint32_t bq[NBC][2 * NG][2];
    float qs[NBC][NG][2];  // sum over group of the f16 (scaled) q, heads 2c and 2c+1
    float qo[NBC][KB == 4 ? NG : 1][2];  // 4-bit keys: the code offsets' share of the QK^T dot
    float ie[NBC][2];      // per head: 2^-e * softmax_scale * log2(e)
#pragma unroll
    for (int nb = 0; nb < NBC; ++nb) {
        // columns past the last q-head are padding (a whole block of them past the
        // last block): they repeat head G-1 (MMA columns never mix) and their
        // partials are never written
        const int gq = kG * (hb0 + nb) + g;
        const uint16_t *qrow = p.q + ((int64_t)b * p.QH + (int64_t)h * p.G + (gq < p.G ? gq : p.G - 1)) * D;
        float qv[NG][8];
        float qoff[NG];
        float mx = 0.0f;
#pragma unroll
        for (int G = 0; G < NG; ++G) {
            const uint4 w = *reinterpret_cast<const uint4 *>(qrow + 32 * G + 8 * c);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qv[G][2 * i] = bf16_lo(ww[i]);
                qv[G][2 * i + 1] = bf16_hi(ww[i]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(qv[G][i]));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // power-of-two scale so the largest |q| of the head lands in [2^14, 2^15)
        int e = 0;
        if (mx > 0.0f && mx < INFINITY) e = 14 - (((int)(__float_as_uint(mx) >> 23) & 0xFF) - 127);
        e = e < -100 ? -100 : (e > 100 ? 100 : e);
        const float qscale = ldexpf(1.0f, e);
        float qsum[NG];
#pragma unroll
        for (int G = 0; G < NG; ++G) {
            float f[8];
            uint32_t hw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                hw[i] = pack_f16x2(qv[G][2 * i] * qscale, qv[G][2 * i + 1] * qscale);
                const __half2 hv = *reinterpret_cast<const __half2 *>(&hw[i]);
                f[2 * i] = __low2float(hv);
                f[2 * i + 1] = __high2float(hv);
            }
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) s += f[i];
            qsum[G] = s;
            if constexpr (KB == 8) {
                // a word holds dims 8c+{0..3} (then {4..7}); its bytes pair as (0, 2), (1, 3)
                auto pr = [&](int i, int j) { return pack_f16x2(f[i], f[j]); };
                bq[nb][2 * G][0] = pr(0, 2);
                bq[nb][2 * G][1] = pr(1, 3);
                bq[nb][2 * G + 1][0] = pr(4, 6);
                bq[nb][2 * G + 1][1] = pr(5, 7);
            } else {
                // nibble k of the word = dim 8c+k; unpacked pairs are (k, k+4).  Odd
                // nibbles are read in place (1024 + 16 code), so their q is taken / 16
                auto pr = [&](int i, int j) { return pack_f16x2(f[i], f[j]); };
                auto pr16 = [&](int i, int j) { return pack_f16x2(f[i] * 0.0625f, f[j] * 0.0625f); };
                bq[nb][2 * G][0] = pr(0, 4);
                bq[nb][2 * G][1] = pr16(1, 5);
                bq[nb][2 * G + 1][0] = pr(2, 6);
                bq[nb][2 * G + 1][1] = pr16(3, 7);
                // the 1024 of every key element times the q it meets in the MMA
                const __half2 h1 = *reinterpret_cast<const __half2 *>(&bq[nb][2 * G][1]);
                const __half2 h3 = *reinterpret_cast<const __half2 *>(&bq[nb][2 * G + 1][1]);
                const float so = __low2float(h1) + __high2float(h1) + __low2float(h3) + __high2float(h3);
                qoff[G] = 1024.0f * (f[0] + f[2] + f[4] + f[6] + so);
            }
        }
        // group sums per head: head g lives in lanes 4g..4g+3; gather heads 2c, 2c+1
#pragma unroll
        for (int G = 0; G < NG; ++G) {
            float s = qsum[G];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            qs[nb][G][0] = __shfl_sync(0xffffffffu, s, (2 * c) * 4);
            qs[nb][G][1] = __shfl_sync(0xffffffffu, s, (2 * c + 1) * 4);
            if constexpr (KB == 4) {
                float so = qoff[G];
                so += __shfl_xor_sync(0xffffffffu, so, 1);
                so += __shfl_xor_sync(0xffffffffu, so, 2);
                qo[nb][G][0] = -__shfl_sync(0xffffffffu, so, (2 * c) * 4);
                qo[nb][G][1] = -__shfl_sync(0xffffffffu, so, (2 * c + 1) * 4);
            }
        }
        const float my_ie = ldexpf(1.0f, -e) * p.scale_log2;
        ie[nb][0] = __shfl_sync(0xffffffffu, my_ie, (2 * c) * 4);
        ie[nb][1] = __shfl_sync(0xffffffffu, my_ie, (2 * c + 1) * 4);
    }

    float o[NBC][2 * NG][4];
    float m_run[NBC][2], l_run[NBC][2];
#pragma unroll
    for (int nb = 0; nb < NBC; ++nb) {
#pragma unroll
        for (int i = 0; i < 2 * NG; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) o[nb][i][j] = 0.0f;
        m_run[nb][0] = m_run[nb][1] = -INFINITY;
        l_run[nb][0] = l_run[nb][1] = 0.0f;
    }

    // V field extraction: lane g owns dims 32G + 4g + {0..3}: 4 VB bits at bit
    // (32G + 4g) VB of the row (word 32G VB / 32 + v_word, shift v_shift)
    const int v_word = (4 * VB * g) >> 5, v_shift = (4 * VB * g) & 31;
    const int r0 = 16 * warp + g, r1 = r0 + 8;  // key rows of this lane in the warp's first tile
    const int vr[4] = {16 * warp + 2 * c, 16 * warp + 2 * c + 1, 16 * warp + 2 * c + 8, 16 * warp + 2 * c + 9};

    // lane-constant byte offsets in a stage: key bytes of row r0 per group (row r1 is
    // 8 rows on, the next tile 16 kCW rows on, rows SW bytes apart in a box; the
    // swizzle term is the same for all of them), value words of token vr[q] for
    // group 0 (group G is 12 G bytes on).  The swizzle of an SW-byte box row
    // xors the 16-byte chunk index with row % 8 (SW = 128), (row >> 1) % 4
    // (SW = 64) or (row >> 2) % 2 (SW = 32).
    const uint32_t xr = A::SW == 128 ? g : A::SW == 64 ? ((g >> 1) & 3) : ((g >> 2) & 1);
    uint32_t koff[NG];
#pragma unroll
    for (int G = 0; G < NG; ++G) {
        const int off = KB == 8 ? 32 * G + 8 * c : 16 * G + 4 * c;  // the lane's bytes of group G in the row
        const int box = off / A::SW, col = off % A::SW;
        koff[G] = A::OFF_K + box * (A::ST * A::SW) + r0 * A::SW + ((((uint32_t)col >> 4) ^ xr) << 4) + (col & 15);
    }
    uint32_t voff[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) voff[q] = A::OFF_V + vr[q] * A::RBV + 4 * v_word;
    // token offsets within the split fit 32 bits: a split never holds 2^31 rows
    // (136 B per row at the smallest width would take 292 GB)
    const int split_rows = (int)(t_end - t_begin);
    const uint32_t ring0 = smem_addr(stages);
    bool ok = true;
    int slot = 0;
    uint32_t phase = 0;  // ring slot and barrier parity of stage s
    for (int s = 0; s < n_stages; ++s) {
        if (!mbar_wait_bounded(full0 + 8 * slot, phase, p.err)) {
            ok = false;
            break;
        }
        const uint32_t st = ring0 + slot * A::STAGE;
        // two 16-row tiles per warp and stage (rows 16 warp and 16 kCW + 16 warp): Q K^T for
        // both, one softmax step over both, P V for both; the tile loops are unrolled so
        // the compiler interleaves the tiles' independent chains
        float S[NBC][A::TILES][2][2];  // scores: [block][tile][row g, row g + 8][head 2c, 2c + 1]
#pragma unroll
        for (int t2 = 0; t2 < A::TILES; ++t2) {
            const int tile_r = s * A::ST + (16 * kCW) * t2 + 16 * warp;  // tile's first row from the split's start

            // ---------------- S = Q K^T for 16 tokens x 8 heads per block, per key group
            float acc[NBC][NG][4];
#pragma unroll
            for (int nb = 0; nb < NBC; ++nb)
#pragma unroll
                for (int G = 0; G < NG; ++G)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[nb][G][j] = 0.0f;
#pragma unroll
            for (int G = 0; G < NG; ++G) {
                uint32_t ka[2][4];  // A fragments of the group's two k-steps, shared by the blocks
                if constexpr (KB == 8) {
                    const uint2 k0 = lds64(st + koff[G] + t2 * ((16 * kCW) * A::SW));
                    const uint2 k1 = lds64(st + koff[G] + t2 * ((16 * kCW) * A::SW) + 8 * A::SW);
                    // bytes 0 and 2 (then 1 and 3) of a word -> f16 (1024 + (byte ^ 0x80)):
                    // dims (8c+0, 8c+2), (8c+1, 8c+3), then +4
                    ka[0][0] = kcvt(k0.x, p); ka[0][1] = kcvt(k1.x, p);
                    ka[0][2] = kcvt(shr_fma<8>(k0.x), p); ka[0][3] = kcvt(shr_fma<8>(k1.x), p);
                    ka[1][0] = kcvt(k0.y, p); ka[1][1] = kcvt(k1.y, p);
                    ka[1][2] = kcvt(shr_fma<8>(k0.y), p); ka[1][3] = kcvt(shr_fma<8>(k1.y), p);
                } else {
                    const uint32_t w0 = lds32(st + koff[G] + t2 * ((16 * kCW) * A::SW));
                    const uint32_t w1 = lds32(st + koff[G] + t2 * ((16 * kCW) * A::SW) + 8 * A::SW);
                    // nibbles k and k+4 -> f16: 1024 + nibble for even k, 1024 + 16 nibble
                    // (read in place) for odd k
                    const uint32_t v0 = shr_fma<8>(w0), v1 = shr_fma<8>(w1);
                    ka[0][0] = kcvt(w0, p); ka[0][1] = kcvt(w1, p);
                    ka[0][2] = (w0 & 0x00F000F0u) | 0x64006400u; ka[0][3] = (w1 & 0x00F000F0u) | 0x64006400u;
                    ka[1][0] = kcvt(v0, p); ka[1][1] = kcvt(v1, p);
                    ka[1][2] = (v0 & 0x00F000F0u) | 0x64006400u; ka[1][3] = (v1 & 0x00F000F0u) | 0x64006400u;
                }
#pragma unroll
                for (int nb = 0; nb < NBC; ++nb) {
                    mma16816(acc[nb][G], ka[0][0], ka[0][1], ka[0][2], ka[0][3], bq[nb][2 * G][0], bq[nb][2 * G][1]);
                    mma16816(acc[nb][G], ka[1][0], ka[1][1], ka[1][2], ka[1][3], bq[nb][2 * G + 1][0],
                             bq[nb][2 * G + 1][1]);
                }
            }
            // per-group affine applied to the scores: S = sum_g scale (acc + (zero - off) qsum),
            // both heads of the lane at once on packed fp32 pairs
            {
                // a row's NG fp16 scales (zero points) are NG / 2 words
                const uint32_t m0 = (r0 + (16 * kCW) * t2) * (NG * 2), m1 = (r1 + (16 * kCW) * t2) * (NG * 2);
                uint32_t sw[2][NG / 2], zw[2][NG / 2];
                lds_words(st + A::OFF_KS + m0, sw[0]);
                lds_words(st + A::OFF_KS + m1, sw[1]);
                lds_words(st + A::OFF_KZ + m0, zw[0]);
                lds_words(st + A::OFF_KZ + m1, zw[1]);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    float2 sacc[NBC];
#pragma unroll
                    for (int nb = 0; nb < NBC; ++nb) sacc[nb] = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int G = 0; G < NG; ++G) {
                        const uint16_t sh = (uint16_t)(sw[i][G >> 1] >> (16 * (G & 1)));
                        const uint16_t zh = (uint16_t)(zw[i][G >> 1] >> (16 * (G & 1)));
                        if constexpr (KB == 8) {
                            const float sc = f16_bits_to_f32(sh), zc = f16_bits_to_f32(zh) - kOffset8;
#pragma unroll
                            for (int nb = 0; nb < NBC; ++nb) {
                                const float2 t = __ffma2_rn(make_float2(zc, zc), make_float2(qs[nb][G][0], qs[nb][G][1]),
                                                            make_float2(acc[nb][G][2 * i], acc[nb][G][2 * i + 1]));
                                sacc[nb] = __ffma2_rn(make_float2(sc, sc), t, sacc[nb]);
                            }
                        } else {
                            const float sc = f16_bits_to_f32(sh), zc = f16_bits_to_f32(zh);
#pragma unroll
                            for (int nb = 0; nb < NBC; ++nb) {
                                const float2 t = __ffma2_rn(make_float2(zc, zc), make_float2(qs[nb][G][0], qs[nb][G][1]),
                                                            make_float2(acc[nb][G][2 * i], acc[nb][G][2 * i + 1]));
                                sacc[nb] = __ffma2_rn(make_float2(sc, sc), __fadd2_rn(t, make_float2(qo[nb][G][0], qo[nb][G][1])),
                                                      sacc[nb]);
                            }
                        }
                    }
#pragma unroll
                    for (int nb = 0; nb < NBC; ++nb) {
                        const float2 sv = __fmul2_rn(sacc[nb], make_float2(ie[nb][0], ie[nb][1]));
                        S[nb][t2][i][0] = sv.x;
                        S[nb][t2][i][1] = sv.y;
                    }
                }
                if (tile_r + 16 > split_rows) {  // ragged tail: mask rows past the range
#pragma unroll
                    for (int nb = 0; nb < NBC; ++nb) {
                        if (tile_r + g >= split_rows) S[nb][t2][0][0] = S[nb][t2][0][1] = -INFINITY;
                        if (tile_r + g + 8 >= split_rows) S[nb][t2][1][0] = S[nb][t2][1][1] = -INFINITY;
                    }
                }
            }
        }
        // ---------------- online softmax (base 2) over the warp's tiles, heads 2c, 2c+1
        // The running max is reduced across the rows only when some lane sees a
        // score above it (or no max exists yet); otherwise the weights are
        // 2^(S - m) with the max unchanged, which is the same arithmetic.
        float pr[NBC][A::TILES][2][2];
#pragma unroll
        for (int nb = 0; nb < NBC; ++nb) {
            bool raise = m_run[nb][0] == -INFINITY || m_run[nb][1] == -INFINITY;
#pragma unroll
            for (int t2 = 0; t2 < A::TILES; ++t2)
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    raise = raise || S[nb][t2][i][0] > m_run[nb][0] || S[nb][t2][i][1] > m_run[nb][1];
            if (__any_sync(0xffffffffu, raise)) {
                float alpha[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float mt = fmaxf(S[nb][0][0][j], S[nb][0][1][j]);
#pragma unroll
                    for (int t2 = 1; t2 < A::TILES; ++t2) mt = fmaxf(mt, fmaxf(S[nb][t2][0][j], S[nb][t2][1][j]));
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
                    const float mn = fmaxf(m_run[nb][j], mt);
                    const float mu = mn == -INFINITY ? 0.0f : mn;
                    alpha[j] = ex2(m_run[nb][j] - mu);
                    m_run[nb][j] = mn;
                    float ls = 0.0f;
#pragma unroll
                    for (int t2 = 0; t2 < A::TILES; ++t2) {
                        pr[nb][t2][0][j] = ex2(S[nb][t2][0][j] - mu);
                        pr[nb][t2][1][j] = ex2(S[nb][t2][1][j] - mu);
                        ls += pr[nb][t2][0][j] + pr[nb][t2][1][j];
                    }
                    l_run[nb][j] = l_run[nb][j] * alpha[j] + ls;
                }
                // o[mt][0, 1] and o[mt][2, 3] are (head 2c, head 2c+1) pairs
                const float2 a2 = make_float2(alpha[0], alpha[1]);
#pragma unroll
                for (int mt2 = 0; mt2 < 2 * NG; ++mt2) {
                    const float2 x = __fmul2_rn(make_float2(o[nb][mt2][0], o[nb][mt2][1]), a2);
                    const float2 y = __fmul2_rn(make_float2(o[nb][mt2][2], o[nb][mt2][3]), a2);
                    o[nb][mt2][0] = x.x;
                    o[nb][mt2][1] = x.y;
                    o[nb][mt2][2] = y.x;
                    o[nb][mt2][3] = y.y;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float ls = 0.0f;
#pragma unroll
                    for (int t2 = 0; t2 < A::TILES; ++t2) {
                        pr[nb][t2][0][j] = ex2(S[nb][t2][0][j] - m_run[nb][j]);
                        pr[nb][t2][1][j] = ex2(S[nb][t2][1][j] - m_run[nb][j]);
                        ls += pr[nb][t2][0][j] + pr[nb][t2][1][j];
                    }
                    l_run[nb][j] += ls;
                }
            }
        }
#pragma unroll
        for (int t2 = 0; t2 < A::TILES; ++t2) {
            const int tile_r = s * A::ST + (16 * kCW) * t2 + 16 * warp;  // tile's first row from the split's start
            // ---------------- P^T as the B operand (tokens x heads), transposed in registers
            uint32_t pt0[NBC], pt1[NBC];
#pragma unroll
            for (int nb = 0; nb < NBC; ++nb) {
                pt0[nb] = movmatrix_trans(pack_f16x2(pr[nb][t2][0][0], pr[nb][t2][0][1]));  // tokens 2c, 2c+1; head g
                pt1[nb] = movmatrix_trans(pack_f16x2(pr[nb][t2][1][0], pr[nb][t2][1][1]));  // tokens 2c+8, 2c+9
            }
            // value scales of this lane's four tokens, NG / 2 words each (zero past the range)
            uint32_t vs[4][NG / 2];
#pragma unroll
            for (int q = 0; q < 4; ++q) lds_words(st + A::OFF_VS + (vr[q] + (16 * kCW) * t2) * (NG * 2), vs[q]);
            if (tile_r + 16 > split_rows) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (tile_r + (vr[q] - 16 * warp) >= split_rows)
#pragma unroll
                        for (int k = 0; k < NG / 2; ++k) vs[q][k] = 0u;
            }
            // ---------------- O^T += V^T P'^T, per value group
#pragma unroll
            for (int G = 0; G < NG; ++G) {
                const uint32_t sel = (G & 1) ? 0x7632u : 0x5410u;
                const uint32_t sp0 = __byte_perm(vs[0][G >> 1], vs[1][G >> 1], sel);
                const uint32_t sp1 = __byte_perm(vs[2][G >> 1], vs[3][G >> 1], sel);
                uint32_t b0[NBC], b1[NBC];
#pragma unroll
                for (int nb = 0; nb < NBC; ++nb) {
                    b0[nb] = hmul2(pt0[nb], sp0);
                    b1[nb] = hmul2(pt1[nb], sp1);
                }
                uint32_t av[2][2][2];  // [token pair][m-tile half][row g, row g+8]
                // the 4 VB-bit field (codes of dims 32G + 4g + 0..3 at bits 0, VB, 2 VB,
                // 3 VB) of the lane's four tokens; bits above 4 VB are don't-care
                uint32_t x[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t base = st + voff[q] + t2 * ((16 * kCW) * A::RBV) + 4 * VB * G;
                    if constexpr (VB == 3)  // 12-bit fields may straddle two words
                        x[q] = __funnelshift_r(lds32(base), lds32(base + 4), v_shift);
                    else  // 8- or 16-bit fields sit inside one word
                        x[q] = lds32(base) >> v_shift;
                }
#pragma unroll
                for (int pr2 = 0; pr2 < 2; ++pr2) {  // token pairs (2c, 2c+1) and (2c+8, 2c+9)
                    if constexpr (VB == 3) {
                        // both tokens' fields side by side (first in bits 0-15), then one
                        // code per nibble: codes r0..r3 of the first token in nibbles
                        // 0..3, of the second in nibbles 4..7
                        const uint32_t w = __byte_perm(x[2 * pr2], x[2 * pr2 + 1], 0x5410u);
                        const uint32_t y = (w & 0x003F003Fu) | ((w & 0x0FC00FC0u) * 4u);
                        // each byte of y holds two codes (bits 0-2, 3-5); adding the upper code
                        // to itself moves it to bits 4-6, and nothing carries out of a byte
                        const uint32_t e = y + (y & 0x38383838u);
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            // selector: codes (r, r+1) of the first token, then of the second
                            const uint32_t sel = __byte_perm(e, 0u, half ? 0x0031u : 0x0020u);
                            const uint32_t lo = prmt(p.tl0, p.tl1, sel);  // low f16 bytes of the 4 centroids
                            const uint32_t hi = prmt(p.th0, p.th1, sel);  // high f16 bytes
                            av[pr2][half][0] = __byte_perm(lo, hi, 0x6240u);  // dim r: (first, second)
                            av[pr2][half][1] = __byte_perm(lo, hi, 0x7351u);  // dim r + 1
                        }
                    } else if constexpr (VB == 2) {
                        // both tokens' bytes side by side; for dim r the two codes (a, b)
                        // pick the f16 pair (c[a], c[b]) out of c0..c3 in one permute:
                        // selector nibbles (2a, 2a+1, 2b, 2b+1)
                        const uint32_t u = __byte_perm(x[2 * pr2], x[2 * pr2 + 1], 0x0040u);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint32_t ab = (u >> (2 * r)) & 0x0303u;
                            av[pr2][r >> 1][r & 1] = prmt(p.tl0, p.tl1, ab * 0x22u + 0x1010u);
                        }
                    } else {
                        // the two tokens' 16-bit fields side by side (a nibble per code);
                        // the table is odd, so a code is a magnitude index (code - 8 for
                        // code >= 8, 7 - code below) and a sign (negative below 8):
                        // t has bit 4i set where code i < 8, m the magnitude indices
                        const uint32_t u = __byte_perm(x[2 * pr2], x[2 * pr2 + 1], 0x5410u);
                        const uint32_t t = (~u >> 3) & 0x11111111u;
                        const uint32_t m = (u ^ (t * 7u)) & 0x77777777u;
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const uint32_t sel = __byte_perm(m, 0u, half ? 0x0031u : 0x0020u);
                            const uint32_t lo = prmt(p.tl0, p.tl1, sel), hi = prmt(p.th0, p.th1, sel);
                            // dim r = 2 half (+1): the two tokens' sign bits (bits 4r and 16 + 4r
                            // of t) moved to the f16 sign positions 15 and 31
                            const int r = 2 * half;
                            av[pr2][half][0] = __byte_perm(lo, hi, 0x6240u) ^ ((t << (15 - 4 * r)) & 0x80008000u);
                            av[pr2][half][1] = __byte_perm(lo, hi, 0x7351u) ^ ((t << (11 - 4 * r)) & 0x80008000u);
                        }
                    }
                }
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int nb = 0; nb < NBC; ++nb)
                        mma16816(o[nb][2 * G + half], av[0][half][0], av[0][half][1], av[1][half][0], av[1][half][1],
                                 b0[nb], b1[nb]);
            }
        }
        // the last warp to finish this stage refills its slot with stage s + kStages
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&done[slot], 1u) == kCW - 1) {
                done[slot] = 0;
                if (s + kStages < n_stages) issue(s + kStages);
            }
        }
        if (++slot == kStages) {
            slot = 0;
            phase ^= 1u;
        }
    }
    __syncthreads();  // every warp is done with the ring before it holds the merge

    // ---------------------------------------------------------------- merge the warps
    // per-lane partial row sums -> per-head sums (lanes with equal c)
#pragma unroll
    for (int nb = 0; nb < NBC; ++nb)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            l_run[nb][j] += __shfl_xor_sync(0xffffffffu, l_run[nb][j], 4);
            l_run[nb][j] += __shfl_xor_sync(0xffffffffu, l_run[nb][j], 8);
            l_run[nb][j] += __shfl_xor_sync(0xffffffffu, l_run[nb][j], 16);
        }
    float *mw = merge + warp * NH * (D + 2);  // [column][D] o, then [column] m, [column] l
#pragma unroll
    for (int nb = 0; nb < NBC; ++nb) {
#pragma unroll
        for (int mt = 0; mt < 2 * NG; ++mt) {
            const int G = mt >> 1, half = mt & 1;
            const int d0 = 32 * G + 4 * g + 2 * half;  // row g -> d0, row g+8 -> d0 + 1
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mw[(kG * nb + 2 * c + j) * D + d0] = o[nb][mt][j];
                mw[(kG * nb + 2 * c + j) * D + d0 + 1] = o[nb][mt][2 + j];
            }
        }
        if (g == 0) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mw[NH * D + kG * nb + 2 * c + j] = ok ? m_run[nb][j] : -INFINITY;
                mw[NH * D + NH + kG * nb + 2 * c + j] = ok ? l_run[nb][j] : 0.0f;
            }
        }
    }
    __syncthreads();
    // items (column, 8 dims), NH x D / 8 of them, over the CTA's threads
    for (int item = threadIdx.x; item < NH * (D / 8); item += kThreads) {
        const int hh = item / (D / 8), d8 = (item % (D / 8)) * 8;
        const int hb = hb0 + hh / kG;
        if (hb >= p.NB) break;  // a padding block (columns are in block order)
        float mmax = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCW; ++w) mmax = fmaxf(mmax, merge[w * NH * (D + 2) + NH * D + hh]);
        const float mu = mmax == -INFINITY ? 0.0f : mmax;
        float ov[8] = {0, 0, 0, 0, 0, 0, 0, 0}, lsum = 0.0f;
#pragma unroll
        for (int w = 0; w < kCW; ++w) {
            const float *m2 = merge + w * NH * (D + 2);
            const float wt = ex2(m2[NH * D + hh] - mu);
            lsum += m2[NH * D + NH + hh] * wt;
#pragma unroll
            for (int i = 0; i < 8; ++i) ov[i] += m2[hh * D + d8 + i] * wt;
        }
        const int64_t pidx = ((((int64_t)b * p.H + h) * p.NB + hb) * p.splits + split) * kG + hh % kG;
        float4 *dst = reinterpret_cast<float4 *>(p.part_o + pidx * D + d8);
        dst[0] = make_float4(ov[0], ov[1], ov[2], ov[3]);
        dst[1] = make_float4(ov[4], ov[5], ov[6], ov[7]);
        if (d8 == 0) {
            p.part_ml[2 * pidx] = mmax;
            p.part_ml[2 * pidx + 1] = lsum;
        }
    }
}

// ---------------------------------------------------------------- combine + deferred un-rotation
struct CombineParams {
    const float *part_o, *part_ml;
    float *out;  // [B][QH][D]
    int H, QH, G, NB, splits, rows;  // rows = B * QH
    float inv_sqrt_d;
    SignBits sg;  // value signs
};

// Each (sequence, q-head) row takes W warps (32 above 128 splits, 16 from 64,
// 4 from 16, else 1, so small merges are not spread thin); a CTA holds
// max(8, W) warps.  Lane holds dims
// 4 lane .. 4 lane + 3.  Warp w of a row merges the splits w, w + W, ...:
// up to kFew of them with every load issued before any is used (one memory
// round trip), more in chunks of 32 whose (max, sum) pairs are read one per
// lane, the weights 2^(m_s - m) computed one per lane and broadcast, and the
// chunk's output rows read with independent loads.  The row's first warp
// then merges its warps' results.
constexpr int kCombineWarps = 8;
constexpr int kFew = 8;
constexpr int kCombD = 128;  // head_dim of this merge (other head_dims take the generic kernel's)

__host__ __device__ constexpr int combine_cta_warps(int W) { return W > kCombineWarps ? W : kCombineWarps; }

template <int W>
__global__ void __launch_bounds__(combine_cta_warps(W) * 32) attn_combine_kernel(const __grid_constant__ CombineParams p)
{
    constexpr int CW = combine_cta_warps(W);
    __shared__ float4 wo[W > 1 ? CW : 1][32];
    __shared__ float wm[CW], wl[CW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * (CW / W) + warp / W, wid = warp % W, lead = warp - wid;
    const bool live = row < p.rows;
    pdl_wait_primary();  // the split kernel's partials are complete and visible
    pdl_allow_dependents();
    if (W == 1 && !live) return;  // no barrier below when W = 1
    const int b = row / p.QH, qh = row % p.QH;
    const int h = qh / p.G, hq = qh % p.G;
    const int hh = hq % kG;  // column of block hq / kG
    const int64_t base = ((int64_t)b * p.H * p.NB + (int64_t)h * p.NB + hq / kG) * p.splits;
    // this warp's splits: wid + W i, i = 0 .. n_mine - 1
    const int n_mine = live && p.splits > wid ? (p.splits - wid + W - 1) / W : 0;
    auto split_index = [&](int i) { return (base + wid + (int64_t)W * i) * kG + hh; };
    float mw = -INFINITY;
    float4 xw = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float lw = 0.0f;
    if (n_mine <= kFew) {
        float2 ml = make_float2(-INFINITY, 0.0f);
        if (lane < n_mine) ml = *reinterpret_cast<const float2 *>(p.part_ml + 2 * split_index(lane));
        float4 v[kFew];
#pragma unroll
        for (int j = 0; j < kFew; ++j)
            v[j] = j < n_mine ? *reinterpret_cast<const float4 *>(p.part_o + split_index(j) * kCombD + 4 * lane)
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        mw = ml.x;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
        const float muw = mw == -INFINITY ? 0.0f : mw;
        const float wt = lane < n_mine ? ex2(ml.x - muw) : 0.0f;
        if (lane < n_mine) lw = ml.y * wt;
#pragma unroll
        for (int j = 0; j < kFew; ++j) {
            const float w = __shfl_sync(0xffffffffu, wt, j);
            xw.x += v[j].x * w; xw.y += v[j].y * w; xw.z += v[j].z * w; xw.w += v[j].w * w;
        }
    } else {
        for (int i = lane; i < n_mine; i += 32) mw = fmaxf(mw, p.part_ml[2 * split_index(i)]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
        const float muw = mw == -INFINITY ? 0.0f : mw;
        for (int i0 = 0; i0 < n_mine; i0 += 32) {
            // lane j: weight and sum of split i0 + j
            float wt = 0.0f;
            if (i0 + lane < n_mine) {
                const float2 ml = *reinterpret_cast<const float2 *>(p.part_ml + 2 * split_index(i0 + lane));
                wt = ex2(ml.x - muw);
                lw += ml.y * wt;
            }
            const int cnt = n_mine - i0 < 32 ? n_mine - i0 : 32;
#pragma unroll 8
            for (int j = 0; j < cnt; ++j) {
                const float w = __shfl_sync(0xffffffffu, wt, j);
                const float4 v = *reinterpret_cast<const float4 *>(p.part_o + split_index(i0 + j) * kCombD + 4 * lane);
                xw.x += v.x * w; xw.y += v.y * w; xw.z += v.z * w; xw.w += v.w * w;
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
    float x[4] = {xw.x, xw.y, xw.z, xw.w}, l = lw;
    if constexpr (W > 1) {
        wo[warp][lane] = xw;
        if (lane == 0) {
            wm[warp] = mw;
            wl[warp] = lw;
        }
        __syncthreads();
        if (wid != 0 || !live) return;
        float mmax = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) mmax = fmaxf(mmax, wm[lead + w]);
        const float mu = mmax == -INFINITY ? 0.0f : mmax;
        l = 0.0f;
        x[0] = x[1] = x[2] = x[3] = 0.0f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            // a warp without live splits carries zeros; the others rescale to the common max
            const float wt = wm[lead + w] == -INFINITY ? 0.0f : ex2(wm[lead + w] - mu);
            l += wl[lead + w] * wt;
            const float4 v = wo[lead + w][lane];
            x[0] += v.x * wt; x[1] += v.y * wt; x[2] += v.z * wt; x[3] += v.w * wt;
        }
    }
    const float inv_l = 1.0f / l;
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] *= inv_l;
    // inverse transform: 2 stages in-lane, 5 across lanes (Sylvester order)
#pragma unroll
    for (int hs = 1; hs < 4; hs <<= 1)
#pragma unroll
        for (int i = 0; i < 4; i += 2 * hs)
#pragma unroll
            for (int j = i; j < i + hs; ++j) {
                const float a = x[j], bb = x[j + hs];
                x[j] = a + bb;
                x[j + hs] = a - bb;
            }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, x[i], m);
            x[i] = upper ? other - x[i] : x[i] + other;
        }
    }
    float4 r;
    float *rr = &r.x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int dim = 4 * lane + i;
        const bool neg = sign_negative(p.sg, dim);
        rr[i] = x[i] * (neg ? -p.inv_sqrt_d : p.inv_sqrt_d);
    }
    *reinterpret_cast<float4 *>(p.out + ((int64_t)b * p.QH + qh) * kCombD + 4 * lane) = r;
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tensor_map_encoder(); }

struct SplitPlan {
    int splits;
    int64_t tokens_per_split;
};

SplitPlan plan_splits(int B, int H, int64_t seq_len, int ctas_per_sm, int stage_t)
{
    const int64_t units = (int64_t)B * H;
    const int64_t stages = (seq_len + stage_t - 1) / stage_t;
    const int64_t slots = (int64_t)num_sms() * ctas_per_sm;
    SplitPlan best{1, stages * stage_t};
    double best_cost = 1e300;
    for (int waves = 1; waves <= 16; ++waves) {
        int64_t s = (waves * slots + units - 1) / units;
        if (s < 1) s = 1;
        if (s > stages) s = stages;
        const int64_t per = (stages + s - 1) / s;  // stages per split
        const int64_t sp = (stages + per - 1) / per;
        const int64_t ctas = units * sp;
        const double cost = (double)((ctas + slots - 1) / slots) * (double)(per + 2);  // +2: fixed cost per CTA
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = SplitPlan{(int)sp, per * stage_t};
        }
    }
    return best;
}

template <int KB, int D, int VB, int NBC>
int ctas_per_sm_for()
{
    static int cached = 0;  // same on every GB300; only a successful query is kept
    if (!cached) {
        int n = 0;
        if (cudaFuncSetAttribute(attn_split_kernel<KB, D, VB, NBC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AGeo<KB, D, VB, NBC>::SMEM) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_split_kernel<KB, D, VB, NBC>, kThreads,
                                                          AGeo<KB, D, VB, NBC>::SMEM) == cudaSuccess &&
            n > 0)
            cached = n;
        else
            return 1;
    }
    return cached;
}

// Launch the split kernel and the combine with a given split plan, the
// partials in `buf` (at least the plan's bytes; see plan_bytes).
template <int KB, int D, int VB, int NBC>
cudaError_t run_attention_plan(const CacheView &c, const uint16_t *q, int QH, int64_t seq_len, float scale, float *out,
                               void *buf, const SplitPlan &plan, cudaStream_t s)
{
    using A = AGeo<KB, D, VB, NBC>;
    if (plan.tokens_per_split % A::ST != 0) return cudaErrorInvalidValue;  // splits start on stage boundaries
    cudaError_t e =
        cudaFuncSetAttribute(attn_split_kernel<KB, D, VB, NBC>, cudaFuncAttributeMaxDynamicSharedMemorySize, A::SMEM);
    if (e != cudaSuccess) return e;
    const size_t need_o = (size_t)c.B * c.H * col_blocks(QH / c.H) * plan.splits * kG * D * 4;

    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)A::KROW, (cuuint64_t)c.B * c.H * c.cap};
    const cuuint64_t gstride[1] = {(cuuint64_t)A::KROW};
    const cuuint32_t box[2] = {(cuuint32_t)A::SW, (cuuint32_t)A::ST};
    const cuuint32_t estride[2] = {1, 1};
    const CUtensorMapSwizzle swz =
        A::SW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : A::SW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c.k_codes, gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
           swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    AttnParams p{};
    p.k_scale = c.k_scale;
    p.k_zero = c.k_zero;
    p.v_scale = c.v_scale;
    p.v_codes = c.v_codes;
    p.q = q;
    p.part_o = static_cast<float *>(buf);
    p.part_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(buf) + need_o);
    p.H = c.H;
    p.QH = QH;
    p.G = QH / c.H;
    p.NB = col_blocks(p.G);
    p.splits = plan.splits;
    p.cap = c.cap;
    p.seq_len = seq_len;
    p.tokens_per_split = plan.tokens_per_split;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = device_error_word();
    if (!p.err) return cudaErrorInvalidDevice;
    const Tables &tab = codebook_tables(VB);
    auto f16b = [](float x) { return (uint32_t)__half_as_ushort(__float2half_rn(x)); };
    if constexpr (VB == 2) {
        p.tl0 = f16b(tab.centroids[0]) | f16b(tab.centroids[1]) << 16;
        p.tl1 = f16b(tab.centroids[2]) | f16b(tab.centroids[3]) << 16;
    } else {
        // 3 bits: the eight centroids; 4 bits: the eight magnitudes c8..c15
        const int first = VB == 3 ? 0 : 8;
        uint32_t lo[8], hi[8];
        for (int i = 0; i < 8; ++i) {
            const uint32_t hb = f16b(tab.centroids[first + i]);
            lo[i] = hb & 0xFF;
            hi[i] = hb >> 8;
        }
        p.tl0 = lo[0] | lo[1] << 8 | lo[2] << 16 | lo[3] << 24;
        p.tl1 = lo[4] | lo[5] << 8 | lo[6] << 16 | lo[7] << 24;
        p.th0 = hi[0] | hi[1] << 8 | hi[2] << 16 | hi[3] << 24;
        p.th1 = hi[4] | hi[5] << 8 | hi[6] << 16 | hi[7] << 24;
    }
    // bits where R1 is set take R2; the others take byte ^ R2 (flip bit 7 and 23)
    p.k_const = KB == 8 ? 0xFF00FF00u : 0xFFF0FFF0u;
    p.k_flip = KB == 8 ? 0x64806480u : 0x64006400u;

    dim3 grid(plan.splits, c.H * ((p.NB + NBC - 1) / NBC), c.B);
    e = launch_dependent(attn_split_kernel<KB, D, VB, NBC>, grid, dim3(kThreads), A::SMEM, s, map, p);
    if (e != cudaSuccess) return e;
    if constexpr (D != kCombD)  // the generic kernel's merge: the same partial layout (one query row)
        return launch_attention_combine_parts(D, p.part_o, p.part_ml, out, c.B, c.H, QH, 1, p.NB, kG, plan.splits,
                                              c.signs, s);

    CombineParams cp{};
    cp.part_o = p.part_o;
    cp.part_ml = p.part_ml;
    cp.out = out;
    cp.H = c.H;
    cp.QH = QH;
    cp.G = QH / c.H;
    cp.NB = col_blocks(cp.G);
    cp.rows = c.B * QH;
    cp.splits = plan.splits;
    cp.inv_sqrt_d = inv_sqrt_head_dim(kCombD);
    cp.sg = c.signs;
    // the merge is a programmatic dependent of the split kernel: its CTAs take
    // SMs as split CTAs retire and wait for the whole split grid before reading
    const dim3 cb(kCombineWarps * 32);
    if (plan.splits > 128) return launch_dependent(attn_combine_kernel<32>, dim3(cp.rows), dim3(32 * 32), 0, s, cp);
    if (plan.splits >= 64) return launch_dependent(attn_combine_kernel<16>, dim3(cp.rows), dim3(16 * 32), 0, s, cp);
    if (plan.splits >= 16) return launch_dependent(attn_combine_kernel<4>, dim3((cp.rows + 1) / 2), cb, 0, s, cp);
    return launch_dependent(attn_combine_kernel<1>, dim3((cp.rows + 7) / 8), cb, 0, s, cp);
}

// Bytes of the split partials of a plan: (d output sums + max + sum) per
// column of each (sequence, kv-head, column block, split).
size_t plan_bytes(const CacheView &c, int QH, const SplitPlan &plan)
{
    return (size_t)c.B * c.H * col_blocks(QH / c.H) * plan.splits * kG * (c.d + 2) * 4;
}

// Column blocks per CTA: two where a kv-head has more than one block and the
// head_dim is at most 128 (at 256 the doubled registers would not fit), else one.
int blocks_per_cta(const CacheView &c, int QH) { return c.d <= 128 && col_blocks(QH / c.H) >= 2 ? 2 : 1; }

template <int D, int VB, int NBC>
int ctas_per_sm_dvn(const CacheView &c)
{
    return c.kb == 8 ? ctas_per_sm_for<8, D, VB, NBC>() : ctas_per_sm_for<4, D, VB, NBC>();
}

template <int D, int VB>
int ctas_per_sm_dv(const CacheView &c, int nbc)
{
    if constexpr (D <= 128)
        if (nbc == 2) return ctas_per_sm_dvn<D, VB, 2>(c);
    return ctas_per_sm_dvn<D, VB, 1>(c);
}

template <int D>
int ctas_per_sm_d(const CacheView &c, int nbc)
{
    return c.vb == 2 ? ctas_per_sm_dv<D, 2>(c, nbc) : c.vb == 4 ? ctas_per_sm_dv<D, 4>(c, nbc) : ctas_per_sm_dv<D, 3>(c, nbc);
}

int ctas_per_sm(const CacheView &c, int nbc)
{
    return c.d == 64 ? ctas_per_sm_d<64>(c, nbc) : c.d == 256 ? ctas_per_sm_d<256>(c, nbc) : ctas_per_sm_d<128>(c, nbc);
}

// Tokens per stage of the split kernel that serves this cache and group.
// (the stage size depends on the key width, head_dim and column blocks, not
// on the value width)
int stage_rows(const CacheView &c, int QH)
{
    const bool two = blocks_per_cta(c, QH) == 2;
    switch (c.d) {
    case 64:
        if (two) return c.kb == 8 ? AGeo<8, 64, 3, 2>::ST : AGeo<4, 64, 3, 2>::ST;
        return c.kb == 8 ? AGeo<8, 64, 3, 1>::ST : AGeo<4, 64, 3, 1>::ST;
    case 256: return c.kb == 8 ? AGeo<8, 256, 3, 1>::ST : AGeo<4, 256, 3, 1>::ST;
    default:
        if (two) return c.kb == 8 ? AGeo<8, 128, 3, 2>::ST : AGeo<4, 128, 3, 2>::ST;
        return c.kb == 8 ? AGeo<8, 128, 3, 1>::ST : AGeo<4, 128, 3, 1>::ST;
    }
}

SplitPlan usual_plan(const CacheView &c, int QH, int64_t seq_len)
{
    const int nbc = blocks_per_cta(c, QH);
    return plan_splits(c.B, c.H * ((col_blocks(QH / c.H) + nbc - 1) / nbc), seq_len, ctas_per_sm(c, nbc),
                       stage_rows(c, QH));
}

template <int D, int VB>
cudaError_t run_attention_dv(const CacheView &c, const uint16_t *q, int QH, int64_t seq_len, float scale, float *out,
                             void *buf, const SplitPlan &plan, cudaStream_t s)
{
    if constexpr (D <= 128) {
        if (blocks_per_cta(c, QH) == 2) {
            if (c.kb == 8) return run_attention_plan<8, D, VB, 2>(c, q, QH, seq_len, scale, out, buf, plan, s);
            return run_attention_plan<4, D, VB, 2>(c, q, QH, seq_len, scale, out, buf, plan, s);
        }
    }
    if (c.kb == 8) return run_attention_plan<8, D, VB, 1>(c, q, QH, seq_len, scale, out, buf, plan, s);
    return run_attention_plan<4, D, VB, 1>(c, q, QH, seq_len, scale, out, buf, plan, s);
}

template <int D>
cudaError_t run_attention_d(const CacheView &c, const uint16_t *q, int QH, int64_t seq_len, float scale, float *out,
                            void *buf, const SplitPlan &plan, cudaStream_t s)
{
    if (c.vb == 2) return run_attention_dv<D, 2>(c, q, QH, seq_len, scale, out, buf, plan, s);
    if (c.vb == 4) return run_attention_dv<D, 4>(c, q, QH, seq_len, scale, out, buf, plan, s);
    return run_attention_dv<D, 3>(c, q, QH, seq_len, scale, out, buf, plan, s);
}

cudaError_t run_attention(const CacheView &c, const uint16_t *q, int QH, int64_t seq_len, float scale, float *out,
                          void *buf, const SplitPlan &plan, cudaStream_t s)
{
    switch (c.d) {
    case 64: return run_attention_d<64>(c, q, QH, seq_len, scale, out, buf, plan, s);
    case 256: return run_attention_d<256>(c, q, QH, seq_len, scale, out, buf, plan, s);
    default: return run_attention_d<128>(c, q, QH, seq_len, scale, out, buf, plan, s);
    }
}

// The 4-bit lookup reads magnitudes and a sign: the table must be odd
// (c[15 - k] = -c[k], as the optimum for a symmetric density is).
bool four_bit_table_odd()
{
    const Tables &t = codebook_tables(4);
    for (int k = 0; k < 8; ++k)
        if (t.centroids[15 - k] != -t.centroids[k]) return false;
    return true;
}

}  // namespace

bool attention_supported(int d, int kb, int vb, int group)
{
    static const bool odd4 = four_bit_table_odd();
    return (d == 64 || d == 128 || d == 256) && (vb == 3 || vb == 2 || (vb == 4 && odd4)) && group >= 1 &&
           (kb == 8 || kb == 4);
}

size_t attention_workspace_bytes(const CacheView &c, int q_heads, int64_t seq_len)
{
    if (!attention_supported(c.d, c.kb, c.vb, q_heads / c.H)) return 0;
    return plan_bytes(c, q_heads, usual_plan(c, q_heads, seq_len));
}

cudaError_t launch_attention(const CacheView &c, const uint16_t *q, int q_heads, int64_t seq_len, float scale,
                             float *out, void *ws, size_t ws_bytes, cudaStream_t s)
{
    const SplitPlan plan = usual_plan(c, q_heads, seq_len);
    if (ws_bytes < plan_bytes(c, q_heads, plan)) return cudaErrorInvalidValue;
    return run_attention(c, q, q_heads, seq_len, scale, out, ws, plan, s);
}

}  // namespace tq

// ---------------------------------------------------------------- allocation-free variant
// Same kernels as launch_attention, but the split partials live in a fixed
// array that belongs to the library instead of a caller-provided workspace.
namespace tq {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB on every device that loads the library

// Holds the (max, sum, unnormalised output) partials of the splits.  Every
// call overwrites the part it uses before reading it, so nothing here has to
// start at zero; calls that overlap on the GPU share it and would race.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevicesNoAlloc = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevicesNoAlloc];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a stand-in, so the address is looked up once per
// device (with that device current) and cached.
void *noalloc_scratch_address()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNoAlloc) return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
        g_noalloc_ptr[dev] = ptr;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

bool noalloc_fits(const CacheView &c, int q_heads) { return plan_bytes(c, q_heads, SplitPlan{1, 0}) <= kNoAllocScratchBytes; }

cudaError_t launch_attention_noalloc(const CacheView &c, const uint16_t *q, int q_heads, int64_t seq_len, float scale,
                                     float *out, cudaStream_t s)
{
    void *scratch = noalloc_scratch_address();
    if (!scratch) return cudaErrorInvalidSymbol;
    // the usual split plan, with fewer splits if its partials would not fit
    SplitPlan plan = usual_plan(c, q_heads, seq_len);
    const size_t per_split = plan_bytes(c, q_heads, SplitPlan{1, 0});
    const int64_t max_splits = (int64_t)(kNoAllocScratchBytes / per_split);
    if (max_splits < 1) return cudaErrorInvalidValue;
    if (plan.splits > max_splits) {
        const int st = stage_rows(c, q_heads);
        const int64_t stages = (seq_len + st - 1) / st;
        const int64_t per = (stages + max_splits - 1) / max_splits;
        plan = SplitPlan{(int)((stages + per - 1) / per), per * st};
    }
    return run_attention(c, q, q_heads, seq_len, scale, out, scratch, plan, s);
}

}  // namespace tq
