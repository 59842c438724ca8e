// tq_decode.cu -- the fetch dispatch: keys alone take the key kernel; values
// (with or without the keys of the same rows) take the value kernels of
// tq_decode.cuh, one translation unit per head_dim.
#include "tq_decode.cuh"

namespace tq {

cudaError_t launch_decode(const CacheView &c, int64_t t0, int64_t n, bool f32, void *k_out, void *v_out,
                          cudaStream_t s)
{
    if (!v_out)  // keys alone
        return f32 ? key_dispatch<true>(c, t0, n, k_out, s) : key_dispatch<false>(c, t0, n, k_out, s);
    // values, with the keys of the same rows fetched by the same warps
    switch (c.d) {
    case 64: return launch_decode_values_d64(c, t0, n, f32, v_out, k_out, s);
    case 128: return launch_decode_values_d128(c, t0, n, f32, v_out, k_out, s);
    case 256: return launch_decode_values_d256(c, t0, n, f32, v_out, k_out, s);
    case 512: return launch_decode_values_d512(c, t0, n, f32, v_out, k_out, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tq
