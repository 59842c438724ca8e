// tq_encode_d512.cu -- encode kernels instantiated for head_dim 512.
#include "tq_encode.cuh"

namespace tq {
cudaError_t launch_encode_d512(const CacheView &c, const uint16_t *k, const int64_t ks[3], const uint16_t *v,
                             const int64_t vs[3], int64_t t0, int64_t n, cudaStream_t s)
{
    return encode_d<512>(c, k, ks, v, vs, t0, n, s);
}
}  // namespace tq
