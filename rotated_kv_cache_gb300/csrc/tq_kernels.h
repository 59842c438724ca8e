// tq_kernels.h -- internal launch interface between the C ABI and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace tq {

// Output i of SplitMix64 started at `seed` (Steele, Lea & Flood, OOPSLA 2014).
__host__ __device__ constexpr uint64_t splitmix64(uint64_t seed, uint64_t i)
{
    uint64_t z = seed + (i + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// The value sign vector of one cache as bits (bit e % 32 of word e / 32 set
// when sign e is -1): sign e is -1 when the top bit of SplitMix64 output e of
// the cache's seed is set.  Built on the host once per call and passed to the
// kernels by value (head_dim <= 512).
struct SignBits {
    uint32_t w[16];
};

inline SignBits make_sign_bits(uint64_t seed, int d)
{
    SignBits s{};
    for (int e = 0; e < d; ++e)
        if (splitmix64(seed, (uint64_t)e) >> 63) s.w[e >> 5] |= 1u << (e & 31);
    return s;
}

__host__ __device__ __forceinline__ bool sign_negative(const SignBits &s, int e) { return (s.w[e >> 5] >> (e & 31)) & 1u; }

struct CacheView {
    int d, kb, vb, H, B;
    int64_t cap;
    uint8_t *k_codes;
    uint16_t *k_scale, *k_zero;
    uint8_t *v_codes;
    uint16_t *v_scale;
    SignBits signs;  // the cache's value sign vector
};

struct Tables {
    float centroids[256];
    float boundaries[255];
};

// Host-side tables (computed once per width; thread safe).
const Tables &codebook_tables(int vb);
float inv_sqrt_head_dim(int d);  // fl(1/sqrt(d)) rounded from binary64

uint32_t *device_error_word();  // per current device; nullptr on failure

// cuTensorMapEncodeTiled from the driver, or nullptr when unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

cudaError_t launch_encode(const CacheView &c, const uint16_t *k, const int64_t ks[3], const uint16_t *v,
                          const int64_t vs[3], int64_t t0, int64_t n, cudaStream_t s);

#define TQ_DECLARE_PER_D(D)                                                                                  \
    cudaError_t launch_encode_d##D(const CacheView &c, const uint16_t *k, const int64_t ks[3], const uint16_t *v, \
                                   const int64_t vs[3], int64_t t0, int64_t n, cudaStream_t s);                  \
    cudaError_t launch_decode_values_d##D(const CacheView &c, int64_t t0, int64_t n, bool f32, void *out,        \
                                          void *k_out, cudaStream_t s);
TQ_DECLARE_PER_D(64)
TQ_DECLARE_PER_D(128)
TQ_DECLARE_PER_D(256)
TQ_DECLARE_PER_D(512)
#undef TQ_DECLARE_PER_D

// Attention for every head_dim, bit pair and group size (the specialised
// kernel above covers d128, k8/k4, v3, groups of 8).
// M query rows per sequence (q and out [B][M][q_heads][d]); query row i sees
// cache rows [0, seq_len - M + i].  M = 1 is plain decode attention.
size_t attention_generic_workspace_bytes(const CacheView &c, int q_heads, int64_t m, int64_t seq_len);
cudaError_t launch_attention_generic(const CacheView &c, const uint16_t *q, int q_heads, int64_t m, int64_t seq_len,
                                     float scale, float *out, void *ws, size_t ws_bytes, cudaStream_t s);

// Merge split partials (o, m, l) laid out [B][H][hb][splits][cb][d] (+ [..][cb][2])
// into out [B][m][QH][d]: log-sum-exp over splits, then the inverse rotation.
cudaError_t launch_attention_combine_parts(int d, const float *part_o, const float *part_ml, float *out, int B, int H,
                                           int QH, int m, int hb, int cb, int splits, const SignBits &sg,
                                           cudaStream_t s);

// Multi-token attention on the tcgen05 tensor cores: head_dim 64 or 128 with
// at least 128 (query row, q-head) columns per kv-head.
bool attention_tc_applies(const CacheView &c, int q_heads, int64_t m);
size_t attention_tc_workspace_bytes(const CacheView &c, int q_heads, int64_t m, int64_t seq_len);
cudaError_t launch_attention_tc(const CacheView &c, const uint16_t *q, int q_heads, int64_t m, int64_t seq_len,
                                float scale, float *out, void *ws, size_t ws_bytes, cudaStream_t s);

// Deferred fetch, un-rotation and cache row copy / clear (src null: zeros).
cudaError_t launch_decode_rotated(const CacheView &c, int64_t t0, int64_t n, bool f32, void *out, cudaStream_t s);
cudaError_t launch_unrotate(int d, const SignBits &sg, bool in_f32, const void *x, int64_t rows, bool out_f32, void *out,
                            cudaStream_t s);
cudaError_t launch_copy_rows(const CacheView &dst, int64_t dst_t0, const CacheView *src, int64_t src_t0, int64_t n,
                             cudaStream_t s);

cudaError_t launch_decode(const CacheView &c, int64_t t0, int64_t n, bool f32, void *k_out, void *v_out,
                          cudaStream_t s);

bool attention_supported(int d, int kb, int vb, int group);
size_t attention_workspace_bytes(const CacheView &c, int q_heads, int64_t seq_len);
cudaError_t launch_attention(const CacheView &c, const uint16_t *q, int q_heads, int64_t seq_len, float scale,
                             float *out, void *ws, size_t ws_bytes, cudaStream_t s);

int num_sms();

// Allocation-free decode attention: partials in a library-owned device array.
size_t noalloc_scratch_bytes();
bool noalloc_fits(const CacheView &c, int q_heads);
cudaError_t launch_attention_noalloc(const CacheView &c, const uint16_t *q, int q_heads, int64_t seq_len, float scale,
                                     float *out, cudaStream_t s);

}  // namespace tq
