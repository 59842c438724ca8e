// tq_attention_generic.cu -- dispatch of the generic attention kernels
// (tq_attention_generic.cuh) by head_dim; each head_dim's kernels compile in
// their own translation unit.
#include "tq_kernels.h"

namespace tq {

#define TQ_DECLARE_GENERIC(D)                                                                                          \
    cudaError_t launch_attention_generic_d##D(const CacheView &c, const uint16_t *q, int q_heads, int64_t m,          \
                                              int64_t seq_len, float scale, float *out, void *ws, size_t ws_bytes,   \
                                              cudaStream_t s);                                                       \
    size_t attention_generic_workspace_d##D(const CacheView &c, int q_heads, int64_t m, int64_t seq_len);             \
    cudaError_t launch_attention_combine_parts_d##D(const float *part_o, const float *part_ml, float *out, int B,    \
                                                    int H, int QH, int m, int hb, int cb, int splits,                \
                                                    const SignBits &sg, cudaStream_t s);
TQ_DECLARE_GENERIC(64)
TQ_DECLARE_GENERIC(128)
TQ_DECLARE_GENERIC(256)
TQ_DECLARE_GENERIC(512)
#undef TQ_DECLARE_GENERIC

#define TQ_BY_HEAD_DIM(d, call, bad)                                                                                   \
    switch (d) {                                                                                                       \
    case 64: return call(64);                                                                                          \
    case 128: return call(128);                                                                                        \
    case 256: return call(256);                                                                                        \
    case 512: return call(512);                                                                                        \
    default: return bad;                                                                                               \
    }

cudaError_t launch_attention_combine_parts(int d, const float *part_o, const float *part_ml, float *out, int B, int H,
                                           int QH, int m, int hb, int cb, int splits, const SignBits &sg,
                                           cudaStream_t s)
{
#define TQ_CALL(D) launch_attention_combine_parts_d##D(part_o, part_ml, out, B, H, QH, m, hb, cb, splits, sg, s)
    TQ_BY_HEAD_DIM(d, TQ_CALL, cudaErrorInvalidValue)
#undef TQ_CALL
}

size_t attention_generic_workspace_bytes(const CacheView &c, int q_heads, int64_t m, int64_t seq_len)
{
#define TQ_CALL(D) attention_generic_workspace_d##D(c, q_heads, m, seq_len)
    TQ_BY_HEAD_DIM(c.d, TQ_CALL, 0)
#undef TQ_CALL
}

cudaError_t launch_attention_generic(const CacheView &c, const uint16_t *q, int q_heads, int64_t m, int64_t seq_len,
                                     float scale, float *out, void *ws, size_t ws_bytes, cudaStream_t s)
{
#define TQ_CALL(D) launch_attention_generic_d##D(c, q, q_heads, m, seq_len, scale, out, ws, ws_bytes, s)
    TQ_BY_HEAD_DIM(c.d, TQ_CALL, cudaErrorInvalidValue)
#undef TQ_CALL
}

}  // namespace tq
