// tq_api.cu -- the extern "C" entry points declared in include/tq.h: argument
// validation on the host, then one or more kernel launches on the caller's
// stream.  Nothing here allocates, frees or synchronises (tq_device_error
// excepted, which is documented to synchronise).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/tq.h"
#include "tq_common.cuh"
#include "tq_kernels.h"

namespace tq {

__device__ uint32_t g_device_error;  // see tq_device_error()

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_err_ptr[kMaxDevices];
int g_sms[kMaxDevices];

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}
}  // namespace

uint32_t *device_error_word()
{
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<uint32_t *>(p);
    }
    return g_err_ptr[dev];
}

int num_sms()
{
    const int dev = current_device();
    if (dev < 0) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = n > 0 ? n : 1;
    }
    return g_sms[dev];
}

}  // namespace tq

namespace {

bool valid_head_dim(int32_t d) { return d == 64 || d == 128 || d == 256 || d == 512; }
bool valid_kbits(int32_t b) { return b == 2 || b == 4 || b == 5 || b == 8; }
bool valid_vbits(int32_t b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 8; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// the fetch and un-rotation kernels move 32-byte words
bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

tq_status check_cache(const tq_cache *c)
{
    if (!c) return TQ_ERR_NULL;
    if (!valid_head_dim(c->head_dim)) return TQ_ERR_HEAD_DIM;
    if (!valid_kbits(c->k_bits) || !valid_vbits(c->v_bits)) return TQ_ERR_BITS;
    if (c->num_kv_heads < 1 || c->batch < 1 || c->reserved != 0) return TQ_ERR_SHAPE;
    if (c->capacity < 16 || c->capacity % 16 != 0 || c->capacity > (int64_t(1) << 31)) return TQ_ERR_SHAPE;
    if (!c->k_codes || !c->k_scale || !c->k_zero || !c->v_codes || !c->v_scale) return TQ_ERR_NULL;
    if (!aligned16(c->k_codes) || !aligned16(c->k_scale) || !aligned16(c->k_zero) || !aligned16(c->v_codes) ||
        !aligned16(c->v_scale))
        return TQ_ERR_ALIGN;
    return TQ_OK;
}

// The sign mask of (seed, head_dim); the last one built on this thread is kept,
// since one process usually serves a single seed.
const tq::SignBits &sign_bits(uint64_t seed, int d)
{
    thread_local uint64_t k_seed = 0;
    thread_local int k_d = 0;
    thread_local tq::SignBits k_bits{};
    if (k_d != d || k_seed != seed) {
        k_bits = tq::make_sign_bits(seed, d);
        k_seed = seed;
        k_d = d;
    }
    return k_bits;
}

tq::CacheView view(const tq_cache *c)
{
    return tq::CacheView{c->head_dim, c->k_bits,  c->v_bits,  c->num_kv_heads, c->batch,
                         c->capacity, c->k_codes, c->k_scale, c->k_zero,       c->v_codes,
                         c->v_scale,  sign_bits(c->sign_seed, c->head_dim)};
}

tq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

// One warp waits, through the bounded wait of every kernel here, on a barrier
// that nothing will complete (tq_check_wait_timeout): the wait gives up at its
// limit, records the timeout code and the kernel returns.
__global__ void wait_timeout_kernel(uint32_t *err)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t a = tq::smem_addr(&bar);
    if (threadIdx.x == 0) {
        tq::mbar_init(a, 1);
        tq::fence_mbar_init();
    }
    __syncwarp();
    tq::mbar_wait_bounded(a, 0, err);
}

}  // namespace

extern "C" {

const char *tq_status_string(tq_status s)
{
    switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_NULL: return "null pointer";
    case TQ_ERR_HEAD_DIM: return "head_dim must be 64, 128, 256 or 512";
    case TQ_ERR_BITS: return "k_bits must be 2, 4, 5 or 8 and v_bits 2, 3, 4, 5 or 8";
    case TQ_ERR_SHAPE: return "shape, stride or count out of range";
    case TQ_ERR_CAPACITY: return "rows beyond the cache capacity";
    case TQ_ERR_ALIGN: return "pointer or stride not aligned as the call requires";
    case TQ_ERR_WORKSPACE: return "workspace missing or too small";
    case TQ_ERR_CUDA: return "CUDA launch or query failed";
    case TQ_ERR_UNSUPPORTED: return "parameters not covered by this kernel";
    case TQ_ERR_SCRATCH: return "problem too large for the library's built-in 16 MiB scratch";
    }
    return "unknown status";
}

size_t tq_bytes_per_token_head(int32_t d, int32_t kb, int32_t vb)
{
    if (!valid_head_dim(d) || !valid_kbits(kb) || !valid_vbits(vb)) return 0;
    return (size_t)d * kb / 8 + 2 * 2 * (size_t)(d / 32) + (size_t)d * vb / 8 + 2 * (size_t)(d / 32);
}

tq_status tq_plane_bytes(const tq_cache *c, size_t out[5])
{
    if (!c || !out) return TQ_ERR_NULL;
    if (!valid_head_dim(c->head_dim)) return TQ_ERR_HEAD_DIM;
    if (!valid_kbits(c->k_bits) || !valid_vbits(c->v_bits)) return TQ_ERR_BITS;
    if (c->num_kv_heads < 1 || c->batch < 1 || c->capacity < 1) return TQ_ERR_SHAPE;
    const size_t rows = (size_t)c->batch * c->num_kv_heads * (size_t)c->capacity;
    const size_t d = (size_t)c->head_dim;
    out[0] = rows * d * c->k_bits / 8;
    out[1] = rows * (d / 32) * 2;
    out[2] = rows * (d / 32) * 2;
    out[3] = rows * d * c->v_bits / 8;
    out[4] = rows * (d / 32) * 2;
    return TQ_OK;
}

tq_status tq_sign_vector(int32_t d, uint64_t seed, int8_t *out)
{
    if (!out) return TQ_ERR_NULL;
    if (!valid_head_dim(d)) return TQ_ERR_HEAD_DIM;
    const tq::SignBits s = tq::make_sign_bits(seed, d);
    for (int i = 0; i < d; ++i) out[i] = tq::sign_negative(s, i) ? -1 : 1;
    return TQ_OK;
}

tq_status tq_codebook(int32_t vb, float *centroids, float *boundaries)
{
    if (!valid_vbits(vb)) return TQ_ERR_BITS;
    if (!centroids && !boundaries) return TQ_ERR_NULL;
    const tq::Tables &t = tq::codebook_tables(vb);
    for (int i = 0; i < (1 << vb); ++i) {
        if (centroids) centroids[i] = t.centroids[i];
        if (boundaries && i + 1 < (1 << vb)) boundaries[i] = t.boundaries[i];
    }
    return TQ_OK;
}

tq_status tq_encode_append(const tq_cache *c, const void *k, const int64_t ks[3], const void *v,
                           const int64_t vs[3], int64_t t0, int64_t n, tq_stream_t stream)
{
    tq_status st = check_cache(c);
    if (st != TQ_OK) return st;
    if (t0 < 0 || n < 0) return TQ_ERR_SHAPE;
    if (t0 + n > c->capacity) return TQ_ERR_CAPACITY;
    if (n == 0) return TQ_OK;
    if (!k || !v || !ks || !vs) return TQ_ERR_NULL;
    if (!aligned16(k) || !aligned16(v)) return TQ_ERR_ALIGN;
    for (int i = 0; i < 3; ++i) {
        if (ks[i] < 0 || vs[i] < 0) return TQ_ERR_SHAPE;
        if (ks[i] % 8 != 0 || vs[i] % 8 != 0) return TQ_ERR_ALIGN;
    }
    return cuda_status(tq::launch_encode(view(c), static_cast<const uint16_t *>(k), ks,
                                         static_cast<const uint16_t *>(v), vs, t0, n, (cudaStream_t)stream));
}

tq_status tq_decode(const tq_cache *c, int64_t t0, int64_t n, tq_dtype dt, void *k_out, void *v_out,
                    tq_stream_t stream)
{
    tq_status st = check_cache(c);
    if (st != TQ_OK) return st;
    if (t0 < 0 || n < 0) return TQ_ERR_SHAPE;
    if (t0 + n > c->capacity) return TQ_ERR_CAPACITY;
    if (dt != TQ_BF16 && dt != TQ_F32) return TQ_ERR_SHAPE;
    if (n == 0 || (!k_out && !v_out)) return TQ_OK;
    if ((k_out && !aligned32(k_out)) || (v_out && !aligned32(v_out))) return TQ_ERR_ALIGN;
    return cuda_status(tq::launch_decode(view(c), t0, n, dt == TQ_F32, k_out, v_out, (cudaStream_t)stream));
}

tq_status tq_decode_values_rotated(const tq_cache *c, int64_t t0, int64_t n, tq_dtype dt, void *v_out,
                                   tq_stream_t stream)
{
    tq_status st = check_cache(c);
    if (st != TQ_OK) return st;
    if (t0 < 0 || n < 0) return TQ_ERR_SHAPE;
    if (t0 + n > c->capacity) return TQ_ERR_CAPACITY;
    if (dt != TQ_BF16 && dt != TQ_F32) return TQ_ERR_SHAPE;
    if (n == 0) return TQ_OK;
    if (!v_out) return TQ_ERR_NULL;
    if (!aligned32(v_out)) return TQ_ERR_ALIGN;
    return cuda_status(tq::launch_decode_rotated(view(c), t0, n, dt == TQ_F32, v_out, (cudaStream_t)stream));
}

tq_status tq_unrotate(int32_t d, uint64_t sign_seed, tq_dtype in_dt, const void *x, int64_t rows, tq_dtype out_dt,
                      void *out, tq_stream_t stream)
{
    if (!valid_head_dim(d)) return TQ_ERR_HEAD_DIM;
    if ((in_dt != TQ_BF16 && in_dt != TQ_F32) || (out_dt != TQ_BF16 && out_dt != TQ_F32) || rows < 0) return TQ_ERR_SHAPE;
    if (rows == 0) return TQ_OK;
    if (!x || !out) return TQ_ERR_NULL;
    if (!aligned32(x) || !aligned32(out)) return TQ_ERR_ALIGN;
    if (x == out && in_dt != out_dt) return TQ_ERR_SHAPE;  // in place only with equal element sizes
    return cuda_status(tq::launch_unrotate(d, sign_bits(sign_seed, d), in_dt == TQ_F32, x, rows, out_dt == TQ_F32, out,
                                            (cudaStream_t)stream));
}

tq_status tq_cache_copy_rows(const tq_cache *dst, int64_t dst_t0, const tq_cache *src, int64_t src_t0, int64_t n,
                             tq_stream_t stream)
{
    tq_status st = check_cache(dst);
    if (st != TQ_OK) return st;
    st = check_cache(src);
    if (st != TQ_OK) return st;
    if (dst->head_dim != src->head_dim || dst->k_bits != src->k_bits || dst->v_bits != src->v_bits ||
        dst->num_kv_heads != src->num_kv_heads || dst->batch != src->batch || dst->sign_seed != src->sign_seed)
        return TQ_ERR_SHAPE;
    if (dst_t0 < 0 || src_t0 < 0 || n < 0) return TQ_ERR_SHAPE;
    if (dst_t0 + n > dst->capacity || src_t0 + n > src->capacity) return TQ_ERR_CAPACITY;
    if (n == 0) return TQ_OK;
    if (dst->k_codes == src->k_codes) {  // the same cache
        if (dst_t0 == src_t0) return TQ_OK;
        if (dst_t0 < src_t0 + n && src_t0 < dst_t0 + n) return TQ_ERR_SHAPE;
    }
    const tq::CacheView sv = view(src);
    return cuda_status(tq::launch_copy_rows(view(dst), dst_t0, &sv, src_t0, n, (cudaStream_t)stream));
}

tq_status tq_cache_clear_rows(const tq_cache *c, int64_t t0, int64_t n, tq_stream_t stream)
{
    tq_status st = check_cache(c);
    if (st != TQ_OK) return st;
    if (t0 < 0 || n < 0) return TQ_ERR_SHAPE;
    if (t0 + n > c->capacity) return TQ_ERR_CAPACITY;
    if (n == 0) return TQ_OK;
    return cuda_status(tq::launch_copy_rows(view(c), t0, nullptr, 0, n, (cudaStream_t)stream));
}

int tq_attention_supported(int32_t d, int32_t kb, int32_t vb, int32_t group)
{
    return valid_head_dim(d) && valid_kbits(kb) && valid_vbits(vb) && group >= 1 ? 1 : 0;
}

namespace {
// the specialised kernel where it applies, the generic one elsewhere
bool specialised(const tq_cache *c, int32_t q_heads)
{
    return tq::attention_supported(c->head_dim, c->k_bits, c->v_bits, q_heads / c->num_kv_heads);
}

size_t workspace_bytes(const tq_cache *c, int32_t q_heads, int64_t seq_len)
{
    return specialised(c, q_heads) ? tq::attention_workspace_bytes(view(c), q_heads, seq_len)
                                   : tq::attention_generic_workspace_bytes(view(c), q_heads, 1, seq_len);
}
}  // namespace

size_t tq_attention_workspace_bytes(const tq_cache *c, int32_t q_heads, int64_t seq_len)
{
    if (check_cache(c) != TQ_OK || q_heads < 1 || q_heads % c->num_kv_heads != 0 || seq_len < 1 ||
        seq_len > c->capacity)
        return 0;
    return workspace_bytes(c, q_heads, seq_len);
}

tq_status tq_decode_attention(const tq_cache *c, const void *q, int32_t q_heads, int64_t seq_len, float scale,
                              float *out, void *ws, size_t ws_bytes, tq_stream_t stream)
{
    tq_status st = check_cache(c);
    if (st != TQ_OK) return st;
    if (!q || !out) return TQ_ERR_NULL;
    if (q_heads < 1 || q_heads % c->num_kv_heads != 0) return TQ_ERR_SHAPE;
    if (seq_len < 1) return TQ_ERR_SHAPE;
    if (seq_len > c->capacity) return TQ_ERR_CAPACITY;
    if (!aligned16(q) || !aligned16(out)) return TQ_ERR_ALIGN;
    const size_t need = workspace_bytes(c, q_heads, seq_len);
    if (need == 0) return TQ_ERR_CUDA;  // the occupancy query failed
    if (!ws || ws_bytes < need) return TQ_ERR_WORKSPACE;
    if (!aligned16(ws)) return TQ_ERR_ALIGN;
    const uint16_t *qh = static_cast<const uint16_t *>(q);
    if (specialised(c, q_heads))
        return cuda_status(tq::launch_attention(view(c), qh, q_heads, seq_len, scale, out, ws, ws_bytes, (cudaStream_t)stream));
    return cuda_status(
        tq::launch_attention_generic(view(c), qh, q_heads, 1, seq_len, scale, out, ws, ws_bytes, (cudaStream_t)stream));
}

namespace {
tq_status check_multi(const tq_cache *c, int32_t q_heads, int64_t m, int64_t seq_len)
{
    if (q_heads < 1 || q_heads % c->num_kv_heads != 0) return TQ_ERR_SHAPE;
    if (seq_len < 1 || m < 1 || m > seq_len) return TQ_ERR_SHAPE;
    if (seq_len > c->capacity) return TQ_ERR_CAPACITY;
    const int64_t group = q_heads / c->num_kv_heads;
    if ((int64_t)c->batch * m * q_heads > (int64_t(1) << 30)) return TQ_ERR_SHAPE;
    if ((int64_t)c->num_kv_heads * ((m * group + 7) / 8) > 65535) return TQ_ERR_SHAPE;
    return TQ_OK;
}

// wide chunks (at least 128 columns per kv-head, head_dim 64/128) run on the
// tcgen05 kernel, the rest on the generic mma.sync kernel
size_t multi_workspace_bytes(const tq_cache *c, int32_t q_heads, int64_t m, int64_t seq_len)
{
    return tq::attention_tc_applies(view(c), q_heads, m) ? tq::attention_tc_workspace_bytes(view(c), q_heads, m, seq_len)
                                                         : tq::attention_generic_workspace_bytes(view(c), q_heads, m, seq_len);
}
}  // namespace

size_t tq_multi_token_workspace_bytes(const tq_cache *c, int32_t q_heads, int64_t m, int64_t seq_len)
{
    if (check_cache(c) != TQ_OK || check_multi(c, q_heads, m, seq_len) != TQ_OK) return 0;
    return multi_workspace_bytes(c, q_heads, m, seq_len);
}

tq_status tq_multi_token_attention(const tq_cache *c, const void *q, int32_t q_heads, int64_t m, int64_t seq_len,
                                   float scale, float *out, void *ws, size_t ws_bytes, tq_stream_t stream)
{
    tq_status st = check_cache(c);
    if (st != TQ_OK) return st;
    if (!q || !out) return TQ_ERR_NULL;
    st = check_multi(c, q_heads, m, seq_len);
    if (st != TQ_OK) return st;
    if (!aligned16(q) || !aligned16(out)) return TQ_ERR_ALIGN;
    const size_t need = multi_workspace_bytes(c, q_heads, m, seq_len);
    if (need == 0) return TQ_ERR_CUDA;  // the occupancy query failed
    if (!ws || ws_bytes < need) return TQ_ERR_WORKSPACE;
    if (!aligned16(ws)) return TQ_ERR_ALIGN;
    const uint16_t *qh = static_cast<const uint16_t *>(q);
    if (tq::attention_tc_applies(view(c), q_heads, m))
        return cuda_status(
            tq::launch_attention_tc(view(c), qh, q_heads, m, seq_len, scale, out, ws, ws_bytes, (cudaStream_t)stream));
    return cuda_status(
        tq::launch_attention_generic(view(c), qh, q_heads, m, seq_len, scale, out, ws, ws_bytes, (cudaStream_t)stream));
}

tq_status tq_decode_attention_noalloc(const tq_cache *c, const void *q, int32_t q_heads, int64_t seq_len,
                                      float scale, float *out, tq_stream_t stream)
{
    tq_status st = check_cache(c);
    if (st != TQ_OK) return st;
    if (!q || !out) return TQ_ERR_NULL;
    if (q_heads < 1 || q_heads % c->num_kv_heads != 0) return TQ_ERR_SHAPE;
    if (seq_len < 1) return TQ_ERR_SHAPE;
    if (seq_len > c->capacity) return TQ_ERR_CAPACITY;
    if (!aligned16(q) || !aligned16(out)) return TQ_ERR_ALIGN;
    if (!tq::attention_supported(c->head_dim, c->k_bits, c->v_bits, q_heads / c->num_kv_heads))
        return TQ_ERR_UNSUPPORTED;
    if (!tq::noalloc_fits(view(c), q_heads)) return TQ_ERR_SCRATCH;
    return cuda_status(tq::launch_attention_noalloc(view(c), static_cast<const uint16_t *>(q), q_heads, seq_len,
                                                    scale, out, (cudaStream_t)stream));
}

tq_status tq_check_wait_timeout(tq_stream_t stream)
{
    uint32_t *err = tq::device_error_word();
    if (!err) return TQ_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err);
    return cuda_status(cudaGetLastError());
}

tq_status tq_device_error(uint32_t *host_code)
{
    if (!host_code) return TQ_ERR_NULL;
    if (cudaDeviceSynchronize() != cudaSuccess) return TQ_ERR_CUDA;
    uint32_t zero = 0;
    if (cudaMemcpyFromSymbol(host_code, tq::g_device_error, sizeof(uint32_t)) != cudaSuccess) return TQ_ERR_CUDA;
    if (cudaMemcpyToSymbol(tq::g_device_error, &zero, sizeof(uint32_t)) != cudaSuccess) return TQ_ERR_CUDA;
    return TQ_OK;
}

}  // extern "C"
