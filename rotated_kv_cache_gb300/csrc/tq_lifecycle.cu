// tq_lifecycle.cu -- deferred fetch (rotated-domain values, un-rotation of
// vectors formed there) and cache row copy / clear.
//
// Method: mlx-bun "TurboQuant -- rotation-based quantization", Part A,
// "Deferred inverse FWHT" (attention is linear in the values, so the weighted
// sum is formed on centroid[code] * rms rows and un-rotated once per query
// row) and "Architecture in mlx-bun" (groups run along head_dim only, so token
// slices of the packed planes are byte-safe).
//
// GB300 layout.  The rotated fetch is elementwise: a thread expands one
// 32-group, the grid's y axis walks (sequence, kv-head).  The un-rotation uses
// the value fetch's lane layout (64 elements per lane as fp32 pairs, d/64 lanes
// per row) and the same transform, so its result equals the second half of
// the fetch bit for bit.  Copies move 16-byte words where both sides and the
// length allow it, 4-byte words otherwise (every plane row is a multiple of 4
// bytes).
#include "tq_common.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

// ------------------------------------------------------------------ rotated fetch
struct RotParams {
    const uint8_t *codes;
    const uint16_t *scale;
    void *out;
    int64_t cap, t0, n, groups_per_bh, BH;
    int d;
    float cen[256];
};

template <int VB, bool F32>
__global__ void __launch_bounds__(256) rotated_kernel(const __grid_constant__ RotParams p)
{
    __shared__ float scen[1 << VB];
    pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    for (int i = threadIdx.x; i < (1 << VB); i += blockDim.x) scen[i] = p.cen[i];
    __syncthreads();
    const int64_t gi = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (gi >= p.groups_per_bh) return;
    constexpr int A = align_of_bytes(4 * VB);
    for (int64_t bh = blockIdx.y; bh < p.BH; bh += gridDim.y) {
        const int64_t row0 = bh * p.cap + p.t0;  // rows t0.. of one (sequence, kv-head) are contiguous
        uint32_t w[VB], c[32];
        load_words<VB, A>(p.codes + row0 * (p.d * VB / 8) + gi * (4 * VB), w);
        unpack_group<VB>(w, c);
        const float s = f16_bits_to_f32(p.scale[row0 * (p.d / 32) + gi]);
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __fmul_rn(scen[c[j]], s);
        const int64_t o = bh * p.n * p.d + gi * 32;
        if constexpr (F32) {
            float *dst = static_cast<float *>(p.out) + o;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                st_global_v8(dst + 8 * k, __float_as_uint(x[8 * k]), __float_as_uint(x[8 * k + 1]), __float_as_uint(x[8 * k + 2]),
                             __float_as_uint(x[8 * k + 3]), __float_as_uint(x[8 * k + 4]), __float_as_uint(x[8 * k + 5]),
                             __float_as_uint(x[8 * k + 6]), __float_as_uint(x[8 * k + 7]));
        } else {
            uint16_t *dst = static_cast<uint16_t *>(p.out) + o;
#pragma unroll
            for (int k = 0; k < 2; ++k)
                st_global_v8(dst + 16 * k, pack_bf16x2(x[16 * k], x[16 * k + 1]), pack_bf16x2(x[16 * k + 2], x[16 * k + 3]),
                             pack_bf16x2(x[16 * k + 4], x[16 * k + 5]), pack_bf16x2(x[16 * k + 6], x[16 * k + 7]),
                             pack_bf16x2(x[16 * k + 8], x[16 * k + 9]), pack_bf16x2(x[16 * k + 10], x[16 * k + 11]),
                             pack_bf16x2(x[16 * k + 12], x[16 * k + 13]), pack_bf16x2(x[16 * k + 14], x[16 * k + 15]));
        }
    }
}

template <int VB, bool F32>
cudaError_t run_rotated(const CacheView &c, int64_t t0, int64_t n, void *out, cudaStream_t s)
{
    RotParams p{};
    p.codes = c.v_codes;
    p.scale = c.v_scale;
    p.out = out;
    p.cap = c.cap;
    p.t0 = t0;
    p.n = n;
    p.d = c.d;
    p.groups_per_bh = n * (c.d / 32);
    p.BH = (int64_t)c.B * c.H;
    const Tables &tab = codebook_tables(VB);
    for (int i = 0; i < (1 << VB); ++i) p.cen[i] = tab.centroids[i];
    const int64_t bx = (p.groups_per_bh + 255) / 256;
    if (bx >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    return launch_dependent(rotated_kernel<VB, F32>, dim3((unsigned)bx, (unsigned)imin64(p.BH, 65535)), dim3(256), 0, s, p);
}

template <bool F32>
cudaError_t rotated_vb(const CacheView &c, int64_t t0, int64_t n, void *out, cudaStream_t s)
{
    switch (c.vb) {
    case 2: return run_rotated<2, F32>(c, t0, n, out, s);
    case 3: return run_rotated<3, F32>(c, t0, n, out, s);
    case 4: return run_rotated<4, F32>(c, t0, n, out, s);
    case 5: return run_rotated<5, F32>(c, t0, n, out, s);
    case 8: return run_rotated<8, F32>(c, t0, n, out, s);
    }
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ un-rotation
constexpr int kUWarps = 4;

struct UnrotParams {
    const void *x;
    void *out;
    int64_t rows;
    uint32_t items;  // warp tiles, < 2^31
    float inv_sqrt_d;
    SignBits sg;  // value signs
};

template <int D, bool IN_F32, bool OUT_F32>
__global__ void __launch_bounds__(kUWarps * 32) unrotate_kernel(const __grid_constant__ UnrotParams p)
{
    constexpr int LPR = D / 64, ROWS = 32 / LPR;
    __shared__ __align__(16) float2 smul[LPR][34];  // (+-1/sqrt d) of elements (j, j+32) of each part, padded
    pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    for (int i = threadIdx.x; i < LPR * 32; i += blockDim.x) {
        const int part = i >> 5, j = i & 31, e = 64 * part + j;
        smul[part][j] = make_float2(sign_negative(p.sg, e) ? -p.inv_sqrt_d : p.inv_sqrt_d,
                                    sign_negative(p.sg, e + 32) ? -p.inv_sqrt_d : p.inv_sqrt_d);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane % ROWS, part = lane / ROWS;
    for (uint32_t item = blockIdx.x * kUWarps + warp; item < p.items; item += gridDim.x * kUWarps) {
        const int64_t row = (int64_t)item * ROWS + r;
        const bool valid = row < p.rows;
        const int64_t e0 = row * D + 64 * part;  // first element of this lane
        float2 P[32];
        if (valid) {
            // 32-byte loads (x is 32-byte aligned and rows are whole multiples of 32 bytes)
            if constexpr (IN_F32) {
                const float *src = static_cast<const float *>(p.x) + e0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t a[8], b[8];
                    ld_global_v8(src + 8 * k, a);
                    ld_global_v8(src + 32 + 8 * k, b);
#pragma unroll
                    for (int q = 0; q < 8; ++q) P[8 * k + q] = make_float2(__uint_as_float(a[q]), __uint_as_float(b[q]));
                }
            } else {
                const uint16_t *src = static_cast<const uint16_t *>(p.x) + e0;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    uint32_t a[8], b[8];
                    ld_global_v8(src + 16 * k, a);
                    ld_global_v8(src + 32 + 16 * k, b);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        P[16 * k + 2 * q] = make_float2(bf16_lo(a[q]), bf16_lo(b[q]));
                        P[16 * k + 2 * q + 1] = make_float2(bf16_hi(a[q]), bf16_hi(b[q]));
                    }
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) P[j] = make_float2(0.0f, 0.0f);
        }
        fwht_pairs<LPR, ROWS>(P, part);  // every lane of a row joins the cross-lane stages
        if (!valid) continue;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float4 m = *reinterpret_cast<const float4 *>(&smul[part][j]);
            P[j] = __fmul2_rn(P[j], make_float2(m.x, m.y));
            P[j + 1] = __fmul2_rn(P[j + 1], make_float2(m.z, m.w));
        }
        if constexpr (OUT_F32) {
            float *dst = static_cast<float *>(p.out) + e0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 *q = P + 8 * i;
                st_global_v8(dst + 8 * i, __float_as_uint(q[0].x), __float_as_uint(q[1].x), __float_as_uint(q[2].x),
                             __float_as_uint(q[3].x), __float_as_uint(q[4].x), __float_as_uint(q[5].x), __float_as_uint(q[6].x),
                             __float_as_uint(q[7].x));
                st_global_v8(dst + 32 + 8 * i, __float_as_uint(q[0].y), __float_as_uint(q[1].y), __float_as_uint(q[2].y),
                             __float_as_uint(q[3].y), __float_as_uint(q[4].y), __float_as_uint(q[5].y), __float_as_uint(q[6].y),
                             __float_as_uint(q[7].y));
            }
        } else {
            uint16_t *dst = static_cast<uint16_t *>(p.out) + e0;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float2 *q = P + 16 * i;
                st_global_v8(dst + 16 * i, pack_bf16x2(q[0].x, q[1].x), pack_bf16x2(q[2].x, q[3].x), pack_bf16x2(q[4].x, q[5].x),
                             pack_bf16x2(q[6].x, q[7].x), pack_bf16x2(q[8].x, q[9].x), pack_bf16x2(q[10].x, q[11].x),
                             pack_bf16x2(q[12].x, q[13].x), pack_bf16x2(q[14].x, q[15].x));
                st_global_v8(dst + 32 + 16 * i, pack_bf16x2(q[0].y, q[1].y), pack_bf16x2(q[2].y, q[3].y),
                             pack_bf16x2(q[4].y, q[5].y), pack_bf16x2(q[6].y, q[7].y), pack_bf16x2(q[8].y, q[9].y),
                             pack_bf16x2(q[10].y, q[11].y), pack_bf16x2(q[12].y, q[13].y), pack_bf16x2(q[14].y, q[15].y));
            }
        }
    }
}

template <int D, bool IN_F32, bool OUT_F32>
cudaError_t run_unrotate(const SignBits &sg, const void *x, int64_t rows, void *out, cudaStream_t s)
{
    constexpr int ROWS = 32 / (D / 64);
    const int64_t items = (rows + ROWS - 1) / ROWS;
    if (items >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    UnrotParams p{x, out, rows, (uint32_t)items, inv_sqrt_head_dim(D), sg};
    auto kern = unrotate_kernel<D, IN_F32, OUT_F32>;
    static int per_sm = 0;
    if (!per_sm) {
        int k = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k, kern, kUWarps * 32, 0);
        if (e != cudaSuccess) return e;
        per_sm = k > 0 ? k : 1;
    }
    const int grid = (int)imin64((items + kUWarps - 1) / kUWarps, (int64_t)num_sms() * per_sm);
    return launch_dependent(kern, dim3((unsigned)grid), dim3(kUWarps * 32), 0, s, p);
}

template <int D>
cudaError_t unrotate_d(const SignBits &sg, bool in_f32, bool out_f32, const void *x, int64_t rows, void *out,
                       cudaStream_t s)
{
    if (in_f32)
        return out_f32 ? run_unrotate<D, true, true>(sg, x, rows, out, s) : run_unrotate<D, true, false>(sg, x, rows, out, s);
    return out_f32 ? run_unrotate<D, false, true>(sg, x, rows, out, s) : run_unrotate<D, false, false>(sg, x, rows, out, s);
}

// ------------------------------------------------------------------ row copy / clear
struct CopyParams {
    const uint8_t *src[5];  // null: write zeros
    uint8_t *dst[5];
    int64_t row_bytes[5];
    int64_t src_bh_rows, dst_bh_rows;  // rows between (sequence, kv-head) blocks: the capacities
    int64_t src_t0, dst_t0;
    uint32_t words[5];     // words per (sequence, kv-head) segment
    FastDiv div_words[5];
    uint32_t total[5];     // words of the plane over all segments (< 2^31)
    int vec16[5];          // 16-byte words when both sides start 16-byte aligned and the length allows
};

// blockIdx.y = plane; the plane's (segment, word) space is walked grid-stride
__global__ void __launch_bounds__(256) copy_rows_kernel(const __grid_constant__ CopyParams p)
{
    pdl_wait_primary();  // whatever the previous kernel on the stream writes or reads is settled
    pdl_allow_dependents();
    const int plane = blockIdx.y;
    const int64_t rb = p.row_bytes[plane];
    const uint8_t *src_plane = p.src[plane];
    uint8_t *dst_plane = p.dst[plane];
    const uint32_t words = p.words[plane], total = p.total[plane];
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const uint32_t bh = fast_div(i, p.div_words[plane]), w = i - bh * words;
        uint8_t *d = dst_plane + (bh * p.dst_bh_rows + p.dst_t0) * rb;
        if (p.vec16[plane]) {
            const uint4 v = src_plane ? reinterpret_cast<const uint4 *>(src_plane + (bh * p.src_bh_rows + p.src_t0) * rb)[w]
                                      : make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4 *>(d)[w] = v;
        } else {
            const uint32_t v = src_plane ? reinterpret_cast<const uint32_t *>(src_plane + (bh * p.src_bh_rows + p.src_t0) * rb)[w]
                                         : 0u;
            reinterpret_cast<uint32_t *>(d)[w] = v;
        }
    }
}

}  // namespace

cudaError_t launch_decode_rotated(const CacheView &c, int64_t t0, int64_t n, bool f32, void *out, cudaStream_t s)
{
    return f32 ? rotated_vb<true>(c, t0, n, out, s) : rotated_vb<false>(c, t0, n, out, s);
}

cudaError_t launch_unrotate(int d, const SignBits &sg, bool in_f32, const void *x, int64_t rows, bool out_f32, void *out,
                            cudaStream_t s)
{
    switch (d) {
    case 64: return unrotate_d<64>(sg, in_f32, out_f32, x, rows, out, s);
    case 128: return unrotate_d<128>(sg, in_f32, out_f32, x, rows, out, s);
    case 256: return unrotate_d<256>(sg, in_f32, out_f32, x, rows, out, s);
    case 512: return unrotate_d<512>(sg, in_f32, out_f32, x, rows, out, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_copy_rows(const CacheView &dst, int64_t dst_t0, const CacheView *src, int64_t src_t0, int64_t n,
                             cudaStream_t s)
{
    CopyParams p{};
    const int g = dst.d / 32;
    const int64_t rb[5] = {(int64_t)dst.d * dst.kb / 8, 2 * g, 2 * g, (int64_t)dst.d * dst.vb / 8, 2 * g};
    uint8_t *dp[5] = {dst.k_codes, reinterpret_cast<uint8_t *>(dst.k_scale), reinterpret_cast<uint8_t *>(dst.k_zero),
                      dst.v_codes, reinterpret_cast<uint8_t *>(dst.v_scale)};
    const uint8_t *sp[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
    if (src) {
        sp[0] = src->k_codes;
        sp[1] = reinterpret_cast<const uint8_t *>(src->k_scale);
        sp[2] = reinterpret_cast<const uint8_t *>(src->k_zero);
        sp[3] = src->v_codes;
        sp[4] = reinterpret_cast<const uint8_t *>(src->v_scale);
    }
    p.src_bh_rows = src ? src->cap : 0;
    p.dst_bh_rows = dst.cap;
    p.src_t0 = src_t0;
    p.dst_t0 = dst_t0;
    const int64_t BH = (int64_t)dst.B * dst.H;
    int64_t most = 0;
    for (int i = 0; i < 5; ++i) {
        p.src[i] = sp[i];
        p.dst[i] = dp[i];
        p.row_bytes[i] = rb[i];
        // a segment starts at a multiple of cap * rb (cap % 16 == 0) plus t0 * rb
        const bool a = (dst_t0 * rb[i]) % 16 == 0 && (!src || (src_t0 * rb[i]) % 16 == 0) && (n * rb[i]) % 16 == 0;
        p.vec16[i] = a ? 1 : 0;  // every plane row is a multiple of 4 bytes, so 4-byte words always fit
        const int64_t words = n * rb[i] / (a ? 16 : 4), total = words * BH;
        if (words >= (int64_t(1) << 31) || total >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
        p.words[i] = (uint32_t)words;
        p.div_words[i] = make_fastdiv(words > 0 ? (uint32_t)words : 1u);
        p.total[i] = (uint32_t)total;
        most = most > total ? most : total;
    }
    const int64_t blocks = imin64((most + 255) / 256, (int64_t)num_sms() * 8);
    return launch_dependent(copy_rows_kernel, dim3((unsigned)(blocks > 0 ? blocks : 1), 5), dim3(256), 0, s, p);
}

}  // namespace tq
