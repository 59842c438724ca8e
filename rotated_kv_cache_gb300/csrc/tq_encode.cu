// tq_encode.cu -- dispatch of the append/encode kernels by head_dim (the
// kernels themselves are in tq_encode.cuh, one translation unit per head_dim).
#include "tq_kernels.h"

namespace tq {

cudaError_t launch_encode(const CacheView &c, const uint16_t *k, const int64_t ks[3], const uint16_t *v,
                          const int64_t vs[3], int64_t t0, int64_t n, cudaStream_t s)
{
    switch (c.d) {
    case 64: return launch_encode_d64(c, k, ks, v, vs, t0, n, s);
    case 128: return launch_encode_d128(c, k, ks, v, vs, t0, n, s);
    case 256: return launch_encode_d256(c, k, ks, v, vs, t0, n, s);
    case 512: return launch_encode_d512(c, k, ks, v, vs, t0, n, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tq
