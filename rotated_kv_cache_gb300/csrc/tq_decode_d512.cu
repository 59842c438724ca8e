// tq_decode_d512.cu -- value fetch kernels instantiated for head_dim 512.
#include "tq_decode.cuh"

namespace tq {
cudaError_t launch_decode_values_d512(const CacheView &c, int64_t t0, int64_t n, bool f32, void *out, void *k_out,
                                     cudaStream_t s)
{
    return f32 ? value_dispatch_vb<512, true>(c, t0, n, out, k_out, s)
               : value_dispatch_vb<512, false>(c, t0, n, out, k_out, s);
}
}  // namespace tq
