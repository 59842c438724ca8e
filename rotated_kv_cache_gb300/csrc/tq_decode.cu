// tq_decode.cu -- key fetch kernels and the fetch dispatch (value kernels are
// in tq_decode.cuh, one translation unit per head_dim).
#include "tq_decode.cuh"

namespace tq {

cudaError_t launch_decode(const CacheView &c, int64_t t0, int64_t n, bool f32, void *k_out, void *v_out,
                          cudaStream_t s)
{
    cudaError_t e = cudaSuccess;
    if (k_out) e = f32 ? key_dispatch<true>(c, t0, n, k_out, s) : key_dispatch<false>(c, t0, n, k_out, s);
    if (e != cudaSuccess || !v_out) return e;
    switch (c.d) {
    case 64: return launch_decode_values_d64(c, t0, n, f32, v_out, s);
    case 128: return launch_decode_values_d128(c, t0, n, f32, v_out, s);
    case 256: return launch_decode_values_d256(c, t0, n, f32, v_out, s);
    case 512: return launch_decode_values_d512(c, t0, n, f32, v_out, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tq
