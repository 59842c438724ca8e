// tq_common.cuh -- device helpers shared by the codec kernels (sm_103a).
#pragma once
#include <utility>

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_kernels.h"

namespace tq {

// Device error word codes (see tq_device_error()).
constexpr uint32_t kErrWaitTimeout = 1u;

// ---------------------------------------------------------------- formats
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f32_to_f16_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// Two fp32 -> packed bf16x2 (round to nearest even), lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------- PTX: shared memory, mbarrier, bulk copies
__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As above, but a thread whose phase is not complete sleeps in hardware until
// it completes or up to `ns` nanoseconds pass, instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of a barrier, for at most ~2 s of wall time.  The
// waiting thread sleeps in hardware between checks (woken when the phase
// completes), so waiting warps take no issue slots from working ones.  On
// timeout the device error word gets kErrWaitTimeout and false is returned,
// so a lost copy can never hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t *err)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 200000u)) return true;
        if (global_timer_ns() - t0 > 2000000000ull) {
            atomicOr(err, kErrWaitTimeout);
            return false;
        }
    }
}

// Bulk asynchronous copy global -> shared (this CTA), completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Tensor copy of one box of a 4-D tensor map (coordinates innermost first)
// into shared memory, completing on `bar`.  x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *map, int x, int y, int z, int w, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

// Bulk asynchronous copy shared -> global, tracked by the bulk-group counter.
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until the shared-memory sources of all committed bulk stores have been read.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Wait until all committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order generic-proxy shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Programmatic dependent launch.  A kernel launched by launch_dependent may
// start while the kernel before it on the stream is still running, once every
// CTA of that kernel has run pdl_allow_dependents (or exited).  It must run
// pdl_wait_primary before it touches memory the earlier kernel writes or
// reads; that wait returns when the earlier grid has completed and its writes
// are visible.  Without a programmatic dependency both do nothing.
__device__ __forceinline__ void pdl_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kern` as a programmatic dependent of the previous kernel on `s`.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t a, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ---------------------------------------------------------------- vector stores of a lane's words
// Store N 32-bit words to a global address aligned to A bytes (A in {4, 8, 16}).
template <int N, int A>
__device__ __forceinline__ void store_words(void *dst, const uint32_t (&w)[N])
{
    static_assert(A == 4 || A == 8 || A == 16, "alignment");
    if constexpr (A == 16 && N % 4 == 0) {
        uint4 *p = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int i = 0; i < N / 4; ++i) p[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else if constexpr (A >= 8 && N % 2 == 0) {
        uint2 *p = reinterpret_cast<uint2 *>(dst);
#pragma unroll
        for (int i = 0; i < N / 2; ++i) p[i] = make_uint2(w[2 * i], w[2 * i + 1]);
    } else {
        uint32_t *p = reinterpret_cast<uint32_t *>(dst);
#pragma unroll
        for (int i = 0; i < N; ++i) p[i] = w[i];
    }
}

template <int N, int A>
__device__ __forceinline__ void load_words(const void *src, uint32_t (&w)[N])
{
    if constexpr (A == 16 && N % 4 == 0) {
        const uint4 *p = reinterpret_cast<const uint4 *>(src);
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            uint4 v = p[i];
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
    } else if constexpr (A >= 8 && N % 2 == 0) {
        const uint2 *p = reinterpret_cast<const uint2 *>(src);
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            uint2 v = p[i];
            w[2 * i] = v.x; w[2 * i + 1] = v.y;
        }
    } else {
        const uint32_t *p = reinterpret_cast<const uint32_t *>(src);
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = p[i];
    }
}

// One 32-byte store (address 32-byte aligned): a lane fills whole 32-byte
// sectors, so a warp's store moves no partial sectors.
__device__ __forceinline__ void st_global_v8(void *p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                             uint32_t a5, uint32_t a6, uint32_t a7)
{
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(a4),
                 "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}

// 32 bytes from global memory (32-byte aligned) in one access.
__device__ __forceinline__ void ld_global_v8(const void *p, uint32_t (&v)[8])
{
    asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "l"(p));
}

__host__ __device__ constexpr int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// Division by a run-time constant d >= 1 for dividends x < 2^31: q = (x * m) >> sh
// with sh = 31 + ceil(log2 d), m = ceil(2^sh / d) < 2^32 (Granlund & Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994, Thm 4.2).
struct FastDiv {
    uint32_t m, sh;
};

inline FastDiv make_fastdiv(uint32_t d)
{
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint32_t sh = 31 + l;
    return FastDiv{(uint32_t)(((1ull << sh) + d - 1) / d), sh};
}

__device__ __forceinline__ uint32_t fast_div(uint32_t x, FastDiv f) { return (uint32_t)(((uint64_t)x * f.m) >> f.sh); }

// Largest power of two (<= 16) dividing x.
__host__ __device__ constexpr int align_of_bytes(int x) { return (x % 16 == 0) ? 16 : (x % 8 == 0) ? 8 : (x % 4 == 0) ? 4 : (x % 2 == 0) ? 2 : 1; }

// ---------------------------------------------------------------- Walsh-Hadamard transform on fp32 pairs
// a - b, rounded once (b * -1 is exact)
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a); }

// One butterfly stage of stride H over 32 pairs: (a, b) -> (a + b, a - b).
template <int H>
__device__ __forceinline__ void bfly_stage(float2 (&P)[32])
{
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        const int j = (t / H) * 2 * H + t % H;
        const float2 s = __fadd2_rn(P[j], P[j + H]);
        P[j + H] = fsub2(P[j], P[j + H]);
        P[j] = s;
    }
}

// Unnormalised Sylvester transform of a 64*LPR-element row held by LPR lanes
// (lane = part * ROWS + row), each lane holding P[j] = (element 64 part + j,
// element 64 part + j + 32).  Stages run in the definition's order, strides
// 1, 2, 4, ...: 1..16 on pairs, 32 inside each pair, 64.. across the row's
// lanes by shuffle (the lane with the part bit clear keeps a + b, the other
// a - b), so the result is bit-identical to the plain in-order butterfly.
template <int LPR, int ROWS>
__device__ __forceinline__ void fwht_pairs(float2 (&P)[32], int part)
{
    bfly_stage<1>(P);
    bfly_stage<2>(P);
    bfly_stage<4>(P);
    bfly_stage<8>(P);
    bfly_stage<16>(P);
#pragma unroll
    for (int j = 0; j < 32; ++j) P[j] = make_float2(__fadd_rn(P[j].x, P[j].y), __fsub_rn(P[j].x, P[j].y));
#pragma unroll
    for (int s = 1; s < LPR; s <<= 1) {
        const float g = (part & s) ? -1.0f : 1.0f;
        const float2 g2 = make_float2(g, g);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            float2 o;
            o.x = __shfl_xor_sync(0xffffffffu, P[j].x, ROWS * s);
            o.y = __shfl_xor_sync(0xffffffffu, P[j].y, ROWS * s);
            P[j] = __ffma2_rn(P[j], g2, o);
        }
    }
}

// head_dim 128 (two lanes per row): the transform of fwht_pairs with half its
// cross-lane traffic.  Part-1 lanes hold every pair swapped, (element j + 32,
// element j) of their part, so both lanes of a row send their .y in one shuffle.
// Afterwards lane part p holds (element 32 p + j, element 64 + 32 p + j), the
// second negated when p = 1.  Each output is the same operation on the same
// operands as in fwht_pairs, so the results are identical.
template <int ROWS>
__device__ __forceinline__ void fwht_pairs_d128(float2 (&P)[32], int part)
{
    bfly_stage<1>(P);
    bfly_stage<2>(P);
    bfly_stage<4>(P);
    bfly_stage<8>(P);
    bfly_stage<16>(P);
    const float sg = part ? -1.0f : 1.0f;  // stride 32: (x + y, x - y), or (y - x, x + y) on swapped pairs
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float x = P[j].x, y = P[j].y;
        P[j] = make_float2(__fmaf_rn(sg, x, y), __fmaf_rn(-sg, y, x));
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {  // stride 64 across the row's two lanes
        const float o = __shfl_xor_sync(0xffffffffu, P[j].y, ROWS), a = P[j].x;
        P[j] = make_float2(__fadd_rn(a, o), __fsub_rn(a, o));
    }
}

// ---------------------------------------------------------------- bitstream packing of one 32-group
// Codes c[0..31] (each < 2^B) -> B little-endian words: code i at bits [iB, iB+B)
// of the 32B-bit group string.  All shifts are compile-time.
template <int B>
__device__ __forceinline__ void pack_group(const uint32_t (&c)[32], uint32_t (&w)[B])
{
#pragma unroll
    for (int k = 0; k < B; ++k) w[k] = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int bit = i * B, word = bit >> 5, off = bit & 31;
        w[word] += c[i] << off;  // fields do not overlap: add == or (one IMAD)
        if (off + B > 32) w[word + 1] += c[i] >> (32 - off);
    }
}

template <int B>
__device__ __forceinline__ void unpack_group(const uint32_t (&w)[B], uint32_t (&c)[32])
{
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int bit = i * B, word = bit >> 5, off = bit & 31;
        uint32_t v = w[word] >> off;
        if (off + B > 32) v |= w[word + 1] << (32 - off);
        c[i] = v & ((1u << B) - 1u);
    }
}

}  // namespace tq
