// tq_attention_tc.cu -- multi-token attention on the fifth-generation tensor
// cores (tcgen05), for chunks wide enough to fill the MMA's 128 rows.
//
// Method: mlx-bun "TurboQuant -- rotation-based quantization", Part A:
// "Algorithm" (key (code + zero) * scale, value centroid[code] * rms),
// "Deferred inverse FWHT" (the weighted sum is formed in the rotated domain
// and un-rotated once per query row), and "Packed-value decode fusion
// investigation" (forward passes appending M = 1, 4 or 128 rows; query row i
// of M sees the cache rows before seq_len - M + i + 1).  Same operation,
// partial layout and combine as the generic kernel; this one runs when a
// kv-head has at least 128 (query row, q-head) columns, where the work is a
// dense contraction (at M = 128 and 8 q-heads per kv-head, 1024 columns).
//
// Design.  A CTA is two warpgroups; each owns 128 columns of one kv-head
// (the MMA's M = 128, one column per tensor-memory lane and per thread) and
// the CTA streams the kv-head's rows of one split in 128-row stages:
//  1. one thread keeps two packed stages in flight with bulk copies
//     completing on mbarriers;
//  2. all 256 threads dequantise the stage into shared memory as f16 MMA
//     operands with 128-byte swizzle: keys as a two-term split
//     k = hi + lo (hi = f16(k), lo = f16(k - hi)), so the scores keep the
//     fp32 key (f16 alone costs ~1e-2 on heavy-tailed keys), K-major; values
//     centroid * rms, MN-major (rows of dims, as stored).  Powers of two
//     keep f16 in range: per key tile, chosen from its group metadata and
//     undone on the scores; one for all value tiles, fixed by the largest
//     finite rms, undone on the output;
//  3. one thread issues S = Q K^T (hi and lo into one accumulator) for both
//     warpgroups into tensor memory and commits to per-warpgroup mbarriers;
//  4. each thread reads its column's 128 scores (tcgen05.ld, 32 at a time,
//     twice: the maximum, then the weights), applies the causal limit,
//     runs the online base-2 softmax in registers and writes its row of P
//     (f16) over its scores in tensor memory (tcgen05.st);
//  5. the warpgroup's first thread issues O_stage = P V into tensor memory
//     (A operand from tensor memory, so P never touches shared memory);
//     each thread adds its row of O_stage into its register accumulator,
//     rescaled by the running maximum.
// The output of a CTA is the per-column (o, m, l) partial; the generic
// kernel's combine merges the splits and un-rotates.  Every wait is bounded
// (mbarrier with a timeout that sets the device error word).
#include <cuda.h>

#include "tq_common.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int tcT = 128;           // cache rows per stage (the QK MMA's N, the PV MMA's K)
constexpr int tcWG = 2;            // warpgroups per CTA
constexpr int tcThreads = 128 * tcWG;
constexpr int tcCB = 128 * tcWG;   // columns per CTA
constexpr int tcRing = 2;          // packed stages in flight

struct TcParams {
    const uint8_t *k_codes, *v_codes;
    const uint16_t *k_scale, *k_zero, *v_scale;
    const uint16_t *q;  // [B][M][QH][D] bf16
    float *part_o;      // [B][H][HB][S][256][D]
    float *part_ml;     // [B][H][HB][S][256][2]
    uint32_t *err;
    int H, QH, G, M, cols, HB, splits, kb, vb;
    int64_t cap, seq_len, tokens_per_split, base0;
    int rbk, rbv, off_ks, off_kz, off_vs, off_v, stage_bytes;
    float scale_log2;   // softmax scale * log2(e)
    float kcmax;        // largest |key code| (127 or 2^kb - 1)
    float vscale;       // 2^ev: every value tile holds centroid * rms * 2^ev
    float cen[256];     // value centroids (fp32)
};

// ---------------------------------------------------------------- tcgen05 / descriptor helpers
// Shared-memory matrix descriptor: 128-byte swizzle, descriptor version 1.
// lbo / sbo in bytes (K-major tiles: sbo = 1024 between 8-row groups, lbo
// unused; MN-major tiles: lbo between 64-element blocks of the M/N extent,
// sbo between 8-row groups of K).
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFF) | (uint64_t)((lbo >> 4) & 0x3FFF) << 16 |
           (uint64_t)((sbo >> 4) & 0x3FFF) << 32 | (uint64_t)1 << 46 | (uint64_t)2 << 61;
}

// Instruction descriptor, kind::f16: f16 A and B, f32 accumulator, M x N,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, int b_mn)
{
    return (1u << 4) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// A operand in tensor memory (M = 128 lanes, two f16 per 32-bit column, the
// even k in the low half), B from shared memory
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's tensor-memory lane
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}


__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

__device__ __forceinline__ float tc_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t tc_pack_f16(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t tc_lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// Byte offset of element (r, k) in a K-major tile of R rows (64-element K blocks
// of R * 128 bytes; 16-byte chunks XOR-swizzled by r % 8).
__host__ __device__ constexpr uint32_t kmaj_off(int R, int r, int k)
{
    return (uint32_t)((k / 64) * (R * 128) + (r / 8) * 1024 + (r % 8) * 128 + ((((k % 64) / 8) ^ (r % 8)) * 16) +
                      (k % 8) * 2);
}

// Byte offset of element (k = cache row, n = dim) of the MN-major value tile
// (N dims: 64-dim blocks 1024 bytes apart inside each group of 8 rows).
template <int N>
__host__ __device__ constexpr uint32_t mnmaj_off(int k, int n)
{
    return (uint32_t)((k / 8) * (N / 64) * 1024 + (n / 64) * 1024 + (k % 8) * 128 + ((((n % 64) / 8) ^ (k % 8)) * 16) +
                      (n % 8) * 2);
}

// power-of-two exponent e with bound * 2^e in [2^13, 2^14) (0 if the bound is
// zero or not finite), clamped to [-100, 100]
__device__ __forceinline__ int tile_exponent(float bound)
{
    if (!(bound > 0.0f) || !(bound < INFINITY)) return 0;
    const int e = 13 - (((int)(__float_as_uint(bound) >> 23) & 0xFF) - 127);
    return e < -100 ? -100 : (e > 100 ? 100 : e);
}

template <int D>
struct TcGeo {
    static constexpr int NG = D / 32;
    static constexpr int KT = tcT * D * 2;     // one key tile (hi or lo): tcT rows x D f16
    static constexpr int VT = tcT * D * 2;     // value tile
    static constexpr int QT = 128 * D * 2;     // one warpgroup's q tile
    static constexpr int OFF_KH = 0, OFF_KL = KT, OFF_V = 2 * KT, OFF_Q = 2 * KT + VT;
    static constexpr int OFF_RING = OFF_Q + tcWG * QT;  // packed stages follow (stage_bytes each)
    static constexpr int SPAN = tcT + D;                 // tensor-memory columns per warpgroup: S (then P), then O
    static constexpr int TMEM_COLS = tcWG * SPAN <= 256 ? 256 : 512;
    static constexpr int WG_COLS = TMEM_COLS / tcWG;
};

// ---------------------------------------------------------------- dequantisation of one 8-element item
// Keys: 8 codes from the 64-bit window (w1:w0) >> sh; kv = (code + zero) * scale * 2^e.
template <int KB>
__device__ __forceinline__ void key_values(uint32_t w0, uint32_t w1, int sh, int kb, float sc, float cz, float (&kv)[8])
{
    uint32_t m[8];
    if constexpr (KB == 8) {
        const uint32_t a = w0 ^ 0x80808080u, b = w1 ^ 0x80808080u;  // int8 -> code + 128
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m[i] = __byte_perm(a, 0x4B000000u, 0x7440 + i);
            m[4 + i] = __byte_perm(b, 0x4B000000u, 0x7440 + i);
        }
    } else if constexpr (KB == 4) {
#pragma unroll
        for (int i = 0; i < 8; ++i) m[i] = ((w0 >> (4 * i)) & 0xFu) | 0x4B000000u;
    } else {
        const uint64_t v = ((uint64_t)w1 << 32 | w0) >> sh;
        const uint32_t mask = (1u << kb) - 1u, flip = kb == 8 ? 0x80u : 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) m[i] = ((((uint32_t)(v >> (i * kb))) & mask) ^ flip) | 0x4B000000u;
    }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const float2 f = __fmul2_rn(fsub2(make_float2(__uint_as_float(m[i]), __uint_as_float(m[i + 1])),
                                          make_float2(cz, cz)),
                                    make_float2(sc, sc));
        kv[i] = f.x;
        kv[i + 1] = f.y;
    }
}

// Values: 8 codes from (w1:w0) >> sh; vv = centroid * rms * 2^ev.
template <int VB>
__device__ __forceinline__ void value_values(uint32_t w0, uint32_t w1, int sh, int vb, float sv, uint32_t lut,
                                             float (&vv)[8])
{
    uint32_t c[8];
    if constexpr (VB == 3) {
        const uint32_t x = __funnelshift_r(w0, w1, sh);
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = (x >> (3 * i)) & 7u;
    } else {
        const uint64_t v = ((uint64_t)w1 << 32 | w0) >> sh;
        const uint32_t mask = (1u << vb) - 1u;
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = (uint32_t)(v >> (i * vb)) & mask;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) vv[i] = __uint_as_float(tc_lds32(lut + 4 * c[i])) * sv;
}

template <int D, int KB, int VB>
__global__ void __launch_bounds__(tcThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams p)
{
    using A = TcGeo<D>;
    pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem + A::OFF_RING;
    float *lut = reinterpret_cast<float *>(ring + tcRing * p.stage_bytes);
    float *red = lut + 256;                                      // per-warp maxima (16 slots)
    uint64_t *bars = reinterpret_cast<uint64_t *>(red + 16);     // full[tcRing], s[2], o[2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + tcRing + 4);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t full0 = smem_addr(bars), bar_s0 = full0 + 8 * tcRing, bar_o0 = bar_s0 + 16;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = tid >> 7, ltid = tid & 127, wq = warp & 3;
    const int split = blockIdx.x, h = blockIdx.y / p.HB, hb = blockIdx.y - h * p.HB, b = blockIdx.z;
    const int64_t bh = (int64_t)b * p.H + h;
    const int col0 = hb * tcCB;
    const int col_last = (p.cols < col0 + tcCB ? p.cols : col0 + tcCB) - 1;
    const int64_t lim_lo = p.base0 + col0 / p.G, lim_hi = p.base0 + col_last / p.G;
    const int64_t t_begin = (int64_t)split * p.tokens_per_split;
    const int64_t t_end = imin64(lim_hi, t_begin + p.tokens_per_split);
    const int n_stages = t_end > t_begin ? (int)((t_end - t_begin + tcT - 1) / tcT) : 0;
    constexpr int NG = A::NG;

    auto issue = [&](int s) {
        const int slot = s % tcRing;
        const int64_t t = t_begin + (int64_t)s * tcT;
        const int rows = (int)imin64(tcT, p.cap - t);
        const int64_t row0 = bh * p.cap + t;
        const uint32_t st = smem_addr(ring + slot * p.stage_bytes), bar = full0 + 8 * slot;
        mbar_arrive_expect_tx(bar, (uint32_t)(rows * (p.rbk + p.rbv + 3 * NG * 2)));
        bulk_g2s(st, p.k_codes + row0 * p.rbk, rows * p.rbk, bar);
        bulk_g2s(st + p.off_ks, p.k_scale + row0 * NG, rows * NG * 2, bar);
        bulk_g2s(st + p.off_kz, p.k_zero + row0 * NG, rows * NG * 2, bar);
        bulk_g2s(st + p.off_vs, p.v_scale + row0 * NG, rows * NG * 2, bar);
        bulk_g2s(st + p.off_v, p.v_codes + row0 * p.rbv, rows * p.rbv, bar);
    };
    int issued = 0;
    if (tid == 0) {
        for (int s = 0; s < tcRing; ++s) mbar_init(full0 + 8 * s, 1);
        for (int w = 0; w < tcWG; ++w) {
            mbar_init(bar_s0 + 8 * w, 1);
            mbar_init(bar_o0 + 8 * w, 1);
        }
        fence_mbar_init();
        for (; issued < tcRing && issued < n_stages; ++issued) issue(issued);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tslot)),
                     "r"(A::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    for (int i = tid; i < (1 << p.vb); i += tcThreads) lut[i] = p.cen[i];

    // ---------------------------------------------------------------- q of this thread's column
    // Scaled by a power of two so its largest |q| lands in [2^14, 2^15): the
    // bf16 values are then exact in f16.  Row ltid of the warpgroup's K-major tile.
    const int col = col0 + 128 * wg + ltid;
    const bool real = col < p.cols;
    const int qi = real ? col / p.G : p.M - 1;
    float ie;
    {
        const int qw = real ? col - qi * p.G : 0;
        const uint16_t *qrow = p.q + (((int64_t)b * p.M + qi) * p.QH + (int64_t)h * p.G + qw) * D;
        float mx = 0.0f;
        if (real)
            for (int c8 = 0; c8 < D / 8; ++c8) {
                const uint4 w = *reinterpret_cast<const uint4 *>(qrow + 8 * c8);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(ww[i])), fabsf(bf16_hi(ww[i]))));
            }
        int e = 0;
        if (mx > 0.0f && mx < INFINITY) e = 14 - (((int)(__float_as_uint(mx) >> 23) & 0xFF) - 127);
        e = e < -100 ? -100 : (e > 100 ? 100 : e);
        const float qs = ldexpf(1.0f, e);
        ie = ldexpf(1.0f, -e) * p.scale_log2;
        const uint32_t qt = sbase + A::OFF_Q + wg * A::QT;
        for (int c8 = 0; c8 < D / 8; ++c8) {
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (real) w = *reinterpret_cast<const uint4 *>(qrow + 8 * c8);
            uint4 hv;
            hv.x = tc_pack_f16(bf16_lo(w.x) * qs, bf16_hi(w.x) * qs);
            hv.y = tc_pack_f16(bf16_lo(w.y) * qs, bf16_hi(w.y) * qs);
            hv.z = tc_pack_f16(bf16_lo(w.z) * qs, bf16_hi(w.z) * qs);
            hv.w = tc_pack_f16(bf16_lo(w.w) * qs, bf16_hi(w.w) * qs);
            sts128(qt + kmaj_off(128, ltid, 8 * c8), hv);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t t_s = tmem + wg * A::WG_COLS, t_o = t_s + tcT;
    const uint32_t t_lane = (uint32_t)(32 * wq) << 16;

    float o[D];
#pragma unroll
    for (int j = 0; j < D; ++j) o[j] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;
    const uint32_t lut_a = smem_addr(lut);
    const float magic_off = p.kb == 8 ? 8388736.0f : 8388608.0f;  // 2^23 (+ 128: int8 codes read as code + 128)
    const int kb = KB ? KB : p.kb, vb = VB ? VB : p.vb;  // compile-time widths for the common schemes

    int s = 0;
    for (; s < n_stages; ++s) {
        const int slot = s % tcRing;
        const bool arrived = mbar_wait_bounded(full0 + 8 * slot, (s / tcRing) & 1, p.err);
        const uint32_t st = smem_addr(ring + slot * p.stage_bytes);
        const int64_t t0 = t_begin + (int64_t)s * tcT;
        const int live = (int)imin64(tcT, t_end - t0);  // rows below t_end

        // ---------------- key tile exponent from the group metadata of the live rows
        // (values use one fixed scale, so their sums can run across stages)
        float bk = 0.0f;
        if (arrived)
            for (int i = tid; i < tcT * NG; i += tcThreads)
                if (i / NG < live) {
                    const float sc = fabsf(f16_bits_to_f32(*reinterpret_cast<const uint16_t *>(ring + slot * p.stage_bytes + p.off_ks + 2 * i)));
                    const float zc = fabsf(f16_bits_to_f32(*reinterpret_cast<const uint16_t *>(ring + slot * p.stage_bytes + p.off_kz + 2 * i)));
                    bk = fmaxf(bk, sc * (zc + p.kcmax));
                }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) bk = fmaxf(bk, __shfl_xor_sync(0xffffffffu, bk, m));
        if (lane == 0) red[warp] = bk;
        if (!__syncthreads_and(arrived && ok)) {
            ok = false;
            break;
        }
        float mk = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) mk = fmaxf(mk, red[w]);
        const int ek = tile_exponent(mk);
        const float sk = ldexpf(1.0f, ek);

        // ---------------- dequantise keys (hi, lo) and values into the operand tiles
        for (int it = tid; it < tcT * (D / 8); it += tcThreads) {
            const int t = it / (D / 8), c8 = it - t * (D / 8), G = c8 >> 2;
            uint4 hi4 = make_uint4(0u, 0u, 0u, 0u), lo4 = hi4, v4 = hi4;
            if (t < live) {
                // keys: 8 codes of kb bits at byte c8 * kb of row t
                const float sc = f16_bits_to_f32(*reinterpret_cast<const uint16_t *>(ring + slot * p.stage_bytes + p.off_ks + 2 * (t * NG + G))) * sk;
                const float zc = f16_bits_to_f32(*reinterpret_cast<const uint16_t *>(ring + slot * p.stage_bytes + p.off_kz + 2 * (t * NG + G)));
                const float cz = magic_off - zc;  // exact: |zero| <= 65504
                const int kbyte = c8 * kb;
                const uint32_t ka = st + t * p.rbk + (kbyte & ~3);
                const uint32_t k0 = tc_lds32(ka), k1 = (kbyte & 3) + kb > 4 ? tc_lds32(ka + 4) : 0u;
                float kv[8];
                key_values<KB>(k0, k1, (kbyte & 3) * 8, kb, sc, cz, kv);
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    hw[i] = tc_pack_f16(kv[2 * i], kv[2 * i + 1]);
                    const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hw[i]));
                    lw[i] = tc_pack_f16(kv[2 * i] - hf.x, kv[2 * i + 1] - hf.y);
                }
                hi4 = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                lo4 = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                // values: 8 codes of vb bits at bit 8 * c8 * vb of row t
                const float sv = f16_bits_to_f32(*reinterpret_cast<const uint16_t *>(ring + slot * p.stage_bytes + p.off_vs + 2 * (t * NG + G))) * p.vscale;
                const int vbit = 8 * c8 * vb;
                const uint32_t va = st + p.off_v + t * p.rbv + 4 * (vbit >> 5);
                const uint32_t v0 = tc_lds32(va), v1 = (vbit & 31) + 8 * vb > 32 ? tc_lds32(va + 4) : 0u;
                float vv[8];
                value_values<VB>(v0, v1, vbit & 31, vb, sv, lut_a, vv);
                v4 = make_uint4(tc_pack_f16(vv[0], vv[1]), tc_pack_f16(vv[2], vv[3]), tc_pack_f16(vv[4], vv[5]),
                                tc_pack_f16(vv[6], vv[7]));
            }
            sts128(sbase + A::OFF_KH + kmaj_off(tcT, t, 8 * c8), hi4);
            sts128(sbase + A::OFF_KL + kmaj_off(tcT, t, 8 * c8), lo4);
            sts128(sbase + A::OFF_V + mnmaj_off<D>(t, 8 * c8), v4);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();  // operands written; the packed slot is free
        tc_fence_after();
        if (tid == 0) {
            if (issued < n_stages) issue(issued++);
            // ---------------- S = Q K^T for both warpgroups (hi then lo into one accumulator)
            constexpr uint32_t idesc_qk = tc_idesc(128, tcT, 0);
#pragma unroll 1
            for (int w = 0; w < tcWG; ++w) {
                const uint32_t qt = sbase + A::OFF_Q + w * A::QT;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ko = (kk / 4) * (tcT * 128) + (kk % 4) * 32;
                    const uint64_t da = tc_desc(qt + (kk / 4) * (128 * 128) + (kk % 4) * 32, 16, 1024);
                    tc_mma(tmem + w * A::WG_COLS, da, tc_desc(sbase + A::OFF_KH + ko, 16, 1024), idesc_qk, kk > 0);
                    tc_mma(tmem + w * A::WG_COLS, da, tc_desc(sbase + A::OFF_KL + ko, 16, 1024), idesc_qk, 1);
                }
                tc_commit(bar_s0 + 8 * w);
            }
        }

        // ---------------- softmax of this thread's column over the stage's rows
        const bool s_done = mbar_wait_bounded(bar_s0 + 8 * wg, s & 1, p.err);
        tc_fence_after();
        // base-2 logits are x * f with f = ie * 2^-ek > 0, so the maximum is taken
        // on x; rows j >= vis are hidden from this query row (this also hides
        // every row at or past t_end)
        const float f = ie * ldexpf(1.0f, -ek);
        const int64_t vis = t0 + tcT > lim_lo ? p.base0 + qi - t0 : (int64_t)tcT;
        // pass 1: the maximum over the stage (32 scores at a time)
        float mt = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < tcT / 32; ++c) {
            uint32_t sr[32];
            tc_ld32(t_s + t_lane + 32 * c, sr);
            tc_wait_ld();
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (32 * c + j < vis) m4[j & 3] = fmaxf(m4[j & 3], __uint_as_float(sr[j]));
            mt = fmaxf(mt, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
        }
        const float mn = fmaxf(m_run, mt * f);
        const float mu = mn == -INFINITY ? 0.0f : mn;
        const float alpha = tc_ex2(m_run - mu);
        m_run = mn;
        // pass 2: the weights; P (f16, two per column) overwrites the row's first
        // tcT / 2 columns in tensor memory, always behind the columns still to
        // be read, and becomes the A operand of P V
        float2 ls = make_float2(0.0f, 0.0f);
#pragma unroll 1
        for (int c = 0; c < tcT / 32; ++c) {
            uint32_t sr[32], pp[16];
            tc_ld32(t_s + t_lane + 32 * c, sr);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float x0 = 32 * c + j < vis ? __uint_as_float(sr[j]) : -INFINITY;
                const float x1 = 32 * c + j + 1 < vis ? __uint_as_float(sr[j + 1]) : -INFINITY;
                const float p0 = tc_ex2(fmaf(x0, f, -mu)), p1 = tc_ex2(fmaf(x1, f, -mu));
                ls = __fadd2_rn(ls, make_float2(p0, p1));
                pp[j / 2] = tc_pack_f16(p0, p1);
            }
            tc_st16(t_s + t_lane + 16 * c, pp);
        }
        tc_wait_st();
        l_run = l_run * alpha + (ls.x + ls.y);
        tc_fence_before();
        named_sync(1 + wg, 128);
        tc_fence_after();
        // ---------------- O_stage = P V (this warpgroup), then o = o * alpha + O_stage
        if (ltid == 0) {
            constexpr uint32_t idesc_pv = tc_idesc(128, D, 1);
            constexpr uint32_t SBO = (D / 64) * 1024;
#pragma unroll
            for (int kk = 0; kk < tcT / 16; ++kk)
                tc_mma_ts(t_o, t_s + kk * 8, tc_desc(sbase + A::OFF_V + kk * 2 * SBO, 1024, SBO), idesc_pv, kk > 0);
            tc_commit(bar_o0 + 8 * wg);
        }
        const bool o_done = mbar_wait_bounded(bar_o0 + 8 * wg, s & 1, p.err);
        tc_fence_after();
        const float2 alpha2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            tc_ld32(t_o + t_lane + 32 * c, orr);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float2 r = __ffma2_rn(make_float2(o[32 * c + j], o[32 * c + j + 1]), alpha2,
                                            make_float2(__uint_as_float(orr[j]), __uint_as_float(orr[j + 1])));
                o[32 * c + j] = r.x;
                o[32 * c + j + 1] = r.y;
            }
        }
        tc_fence_before();
        ok = ok && s_done && o_done;
    }
    // copies still in flight after an early exit: wait for them (bounded)
    if (tid == 0)
        for (int r = s; r < issued; ++r) mbar_wait_bounded(full0 + 8 * (r % tcRing), (r / tcRing) & 1, p.err);

    // ---------------------------------------------------------------- partial of this column
    {
        const int64_t pidx = ((bh * p.HB + hb) * p.splits + split) * tcCB + 128 * wg + ltid;
        float4 *dst = reinterpret_cast<float4 *>(p.part_o + pidx * D);
        const float iv = 1.0f / p.vscale;  // a power of two: exact
#pragma unroll
        for (int i = 0; i < D / 4; ++i)
            dst[i] = make_float4(o[4 * i] * iv, o[4 * i + 1] * iv, o[4 * i + 2] * iv, o[4 * i + 3] * iv);
        p.part_ml[2 * pidx] = ok ? m_run : -INFINITY;
        p.part_ml[2 * pidx + 1] = ok ? l_run : 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(A::TMEM_COLS));
}

// ---------------------------------------------------------------- host side
inline int tile_exponent_host(float bound)
{
    int ex;
    frexpf(bound, &ex);  // bound = f * 2^ex, f in [0.5, 1)
    return 14 - ex;
}

struct TcPlan {
    int hb, splits, stage_bytes, smem;
    int64_t tokens_per_split;
    int off_ks, off_kz, off_vs, off_v;
};

// packed stage layout (key codes, key scales, key zeros, value rms, value
// codes) and the kernel's dynamic shared memory
template <int D>
void tc_layout(int kb, int vb, TcPlan &pl)
{
    const int NG = D / 32, rbk = D * kb / 8, rbv = D * vb / 8;
    auto r16 = [](int x) { return (x + 15) / 16 * 16; };
    pl.off_ks = r16(tcT * rbk);
    pl.off_kz = pl.off_ks + r16(tcT * NG * 2);
    pl.off_vs = pl.off_kz + r16(tcT * NG * 2);
    pl.off_v = pl.off_vs + r16(tcT * NG * 2);
    pl.stage_bytes = (pl.off_v + tcT * rbv + 16 + 127) / 128 * 128;
    pl.smem = 1024 /*align slack*/ + TcGeo<D>::OFF_RING + tcRing * pl.stage_bytes + 256 * 4 /*lut*/ +
              16 * 4 /*maxima*/ + (tcRing + 4) * 8 /*barriers*/ + 16;
}

template <int D, int KB, int VB>
bool tc_plan(const CacheView &c, int q_heads, int64_t m, int64_t seq_len, TcPlan &pl)
{
    using A = TcGeo<D>;
    tc_layout<D>(c.kb, c.vb, pl);
    if (pl.smem > 227 * 1024) return false;
    auto kern = attn_tc_kernel<D, KB, VB>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem) != cudaSuccess) return false;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, tcThreads, pl.smem) != cudaSuccess || per_sm < 1)
        return false;
    // each CTA holds TMEM_COLS of the SM's 512 tensor-memory columns
    if (per_sm * A::TMEM_COLS > 512) per_sm = 512 / A::TMEM_COLS;
    const int64_t cols = (int64_t)(q_heads / c.H) * m;
    pl.hb = (int)((cols + tcCB - 1) / tcCB);
    const int64_t units = (int64_t)c.B * c.H * pl.hb;
    const int64_t nst = (seq_len + tcT - 1) / tcT;
    const int64_t slots = (int64_t)num_sms() * per_sm;
    pl.splits = 1;
    pl.tokens_per_split = nst * tcT;
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
            pl.tokens_per_split = per * tcT;
        }
    }
    return true;
}

template <int D, int KB, int VB>
cudaError_t tc_run(const CacheView &c, const uint16_t *q, int QH, int64_t m, int64_t seq_len, float scale, float *out,
                   void *ws, size_t ws_bytes, cudaStream_t s)
{
    TcPlan pl;
    if (!tc_plan<D, KB, VB>(c, QH, m, seq_len, pl)) return cudaErrorInvalidConfiguration;
    const int G = QH / c.H;
    const size_t parts = (size_t)c.B * c.H * pl.hb * pl.splits * tcCB;
    const size_t need_o = parts * D * 4;
    if (ws_bytes < need_o + parts * 2 * 4) return cudaErrorInvalidValue;
    TcParams p{};
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
    p.scale_log2 = scale * 1.4426950408889634f;
    p.kcmax = c.kb == 8 ? 127.0f : (float)((1 << c.kb) - 1);
    const Tables &tab = codebook_tables(c.vb);
    float cm = 0.0f;
    for (int i = 0; i < (1 << c.vb); ++i) {
        p.cen[i] = tab.centroids[i];
        cm = cm > fabsf(tab.centroids[i]) ? cm : fabsf(tab.centroids[i]);
    }
    // one power of two for every value tile: the largest finite rms (65504)
    // times the largest centroid lands in [2^13, 2^14), so f16 always holds them
    p.vscale = ldexpf(1.0f, tile_exponent_host(65504.0f * cm));
    if ((int64_t)c.H * pl.hb > 65535 || c.B > 65535) return cudaErrorInvalidValue;
    const cudaError_t le = launch_dependent(attn_tc_kernel<D, KB, VB>, dim3(pl.splits, c.H * pl.hb, c.B), dim3(tcThreads), pl.smem, s, p);
    if (le != cudaSuccess) return le;
    return launch_attention_combine_parts(D, p.part_o, p.part_ml, out, c.B, c.H, QH, (int)m, pl.hb, tcCB, pl.splits,
                                          c.signs, s);
}

// compile-time code widths for the common schemes, run-time ones otherwise
template <int D>
cudaError_t tc_dispatch(const CacheView &c, const uint16_t *q, int QH, int64_t m, int64_t seq_len, float scale,
                        float *out, void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (c.kb == 8 && c.vb == 3) return tc_run<D, 8, 3>(c, q, QH, m, seq_len, scale, out, ws, ws_bytes, s);
    if (c.kb == 4 && c.vb == 3) return tc_run<D, 4, 3>(c, q, QH, m, seq_len, scale, out, ws, ws_bytes, s);
    return tc_run<D, 0, 0>(c, q, QH, m, seq_len, scale, out, ws, ws_bytes, s);
}

template <int D>
bool tc_plan_any(const CacheView &c, int q_heads, int64_t m, int64_t seq_len, TcPlan &pl)
{
    if (c.kb == 8 && c.vb == 3) return tc_plan<D, 8, 3>(c, q_heads, m, seq_len, pl);
    if (c.kb == 4 && c.vb == 3) return tc_plan<D, 4, 3>(c, q_heads, m, seq_len, pl);
    return tc_plan<D, 0, 0>(c, q_heads, m, seq_len, pl);
}

}  // namespace

bool attention_tc_applies(const CacheView &c, int q_heads, int64_t m)
{
    if ((c.d != 64 && c.d != 128) || (int64_t)(q_heads / c.H) * m < 128) return false;
    TcPlan pl;  // the packed ring must fit beside the operand tiles
    if (c.d == 64) tc_layout<64>(c.kb, c.vb, pl);
    else tc_layout<128>(c.kb, c.vb, pl);
    return pl.smem <= 227 * 1024;
}

size_t attention_tc_workspace_bytes(const CacheView &c, int q_heads, int64_t m, int64_t seq_len)
{
    TcPlan pl;
    bool ok = c.d == 64 ? tc_plan_any<64>(c, q_heads, m, seq_len, pl) : c.d == 128 ? tc_plan_any<128>(c, q_heads, m, seq_len, pl)
                                                                                 : false;
    if (!ok) return 0;
    return (size_t)c.B * c.H * pl.hb * pl.splits * tcCB * (c.d + 2) * 4;
}

cudaError_t launch_attention_tc(const CacheView &c, const uint16_t *q, int q_heads, int64_t m, int64_t seq_len,
                                float scale, float *out, void *ws, size_t ws_bytes, cudaStream_t s)
{
    switch (c.d) {
    case 64: return tc_dispatch<64>(c, q, q_heads, m, seq_len, scale, out, ws, ws_bytes, s);
    case 128: return tc_dispatch<128>(c, q, q_heads, m, seq_len, scale, out, ws, ws_bytes, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tq
