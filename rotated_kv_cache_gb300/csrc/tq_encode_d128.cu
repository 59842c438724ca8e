// tq_encode_d128.cu -- encode kernels instantiated for head_dim 128.
#include "tq_encode.cuh"

namespace tq {
cudaError_t launch_encode_d128(const CacheView &c, const uint16_t *k, const int64_t ks[3], const uint16_t *v,
                             const int64_t vs[3], int64_t t0, int64_t n, cudaStream_t s)
{
    return encode_d<128>(c, k, ks, v, vs, t0, n, s);
}
}  // namespace tq
