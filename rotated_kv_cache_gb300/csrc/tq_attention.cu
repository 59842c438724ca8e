// tq_attention.cu -- fused dequantise-on-fetch GQA decode attention (placeholder).
#include "tq_kernels.h"

namespace tq {
bool attention_supported(int, int, int, int) { return false; }
size_t attention_workspace_bytes(const CacheView &, int, int64_t) { return 0; }
cudaError_t launch_attention(const CacheView &, const uint16_t *, int, int64_t, float, float *, void *, size_t,
                             cudaStream_t)
{
    return cudaErrorNotSupported;
}
}  // namespace tq
