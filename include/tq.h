/*
 * tq.h -- C ABI of the GB300 (sm_103a) TurboQuant rotated KV-cache codec.
 *
 * The codec is the one defined on the mlx-bun design page "TurboQuant --
 * rotation-based quantization", Part A (KV leg), section "Algorithm
 * (vllm-metal reference semantics, exact)":
 *   keys   -- no rotation; per-32-group asymmetric affine: signed int8 codes
 *             (k_bits = 8) or unsigned 2/4/5-bit codes packed little-endian;
 *             fp16 scale and zero point per group.
 *   values -- x * signs (a fixed +-1 vector), normalised Walsh-Hadamard
 *             transform (1/sqrt(d)), per-32-group RMS scale (fp16), index of
 *             the Lloyd-Max cell of y / (rms + 1e-8), packed little-endian at
 *             v_bits per value.
 * Section "Architecture in mlx-bun" defines dequantize-on-fetch attention
 * (updateAndFetch), and section "Deferred inverse FWHT" the un-rotation of
 * the attention output once per query row, which tq_decode_attention uses.
 *
 * Conventions for every entry point:
 *  - Pointers named *device* are CUDA device memory owned by the caller; the
 *    library never allocates, frees or synchronises.  Host pointers are
 *    read or written before the call returns.
 *  - Arguments are validated on the host before anything is enqueued; a bad
 *    argument returns an error status and enqueues nothing.
 *  - Work is enqueued on `stream` and the call returns; device-side faults
 *    surface at the caller's next synchronisation.  A launch failure returns
 *    TQ_ERR_CUDA.  Calls on one stream are ordered; calls that touch the same
 *    cache rows from different streams must be ordered by the caller.
 *  - The calls other than tq_decode_attention_noalloc are capturable in a
 *    CUDA graph (no allocation, no sync).
 *  - Each kernel is launched as a programmatic dependent of the kernel before
 *    it on the stream and waits for that kernel before it touches memory, so
 *    stream order holds as for ordinary launches; only its start-up overlaps
 *    the previous kernel's end.
 *  - Calls run on the calling thread's current CUDA device, which must hold
 *    every pointer.  The intended use is one process per GPU.  Kernel
 *    shared-memory opt-ins and occupancy figures are set up once per process,
 *    on the first device a kernel runs on; a process that later calls on
 *    another device gets TQ_ERR_CUDA if that device needs its own set-up.
 *    The device error word and the SM count are kept per device.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols of the shared library (the rest is hidden). */
#if defined(__GNUC__)
#define TQ_API __attribute__((visibility("default")))
#else
#define TQ_API
#endif

/* cudaStream_t without including the CUDA headers (same type). */
typedef struct CUstream_st *tq_stream_t;

typedef enum tq_status {
    TQ_OK = 0,
    TQ_ERR_NULL = 1,      /* a required pointer is NULL */
    TQ_ERR_HEAD_DIM = 2,  /* head_dim not in {64, 128, 256, 512} */
    TQ_ERR_BITS = 3,      /* k_bits not in {2,4,5,8} or v_bits not in {2,3,4,5,8} */
    TQ_ERR_SHAPE = 4,     /* batch/heads/tokens/strides out of range */
    TQ_ERR_CAPACITY = 5,  /* rows beyond the cache capacity */
    TQ_ERR_ALIGN = 6,     /* pointer or stride not aligned as the call requires (16 or 32 bytes) */
    TQ_ERR_WORKSPACE = 7, /* workspace missing or too small */
    TQ_ERR_CUDA = 8,      /* a CUDA launch or query failed */
    TQ_ERR_UNSUPPORTED = 9, /* valid codec parameters this kernel does not cover */
    TQ_ERR_SCRATCH = 10     /* too large for the library's built-in scratch (tq_decode_attention_noalloc) */
} tq_status;

typedef enum tq_dtype { TQ_BF16 = 0, TQ_F32 = 1 } tq_dtype;

/*
 * The packed cache: five planes in caller-owned device memory, each laid out
 * [batch][num_kv_heads][capacity][row] row-major, where row is
 *   k_codes  d*k_bits/8 bytes   (int8 two's complement at 8 bits, else the
 *                                little-endian bitstream: code i occupies bits
 *                                [i*b, i*b+b), bit j of the row is bit j%8 of
 *                                byte j/8)
 *   k_scale  d/32 fp16 (IEEE binary16 bit patterns)
 *   k_zero   d/32 fp16
 *   v_codes  d*v_bits/8 bytes   (little-endian bitstream)
 *   v_scale  d/32 fp16
 * Groups of 32 run along head_dim only, so any token range is byte-safe
 * (section "Architecture in mlx-bun" keeps this as a standing rule).  Plane base pointers must
 * be 16-byte aligned and capacity a multiple of 16.
 */
typedef struct tq_cache {
    int32_t head_dim;     /* d in {64, 128, 256, 512} */
    int32_t k_bits;       /* {2, 4, 5, 8} */
    int32_t v_bits;       /* {2, 3, 4, 5, 8} */
    int32_t num_kv_heads; /* H >= 1 */
    int32_t batch;        /* B >= 1 */
    int32_t reserved;     /* must be 0 */
    int64_t capacity;     /* token slots per (sequence, kv-head), multiple of 16 */
    uint8_t *k_codes;     /* device */
    uint16_t *k_scale;    /* device */
    uint16_t *k_zero;     /* device */
    uint8_t *v_codes;     /* device */
    uint16_t *v_scale;    /* device */
    uint64_t sign_seed;   /* seed of the value sign vector (tq_sign_vector); the
                             codec's default is TQ_DEFAULT_SIGN_SEED.  Every call
                             on one cache must use the seed it was encoded with. */
} tq_cache;

/* The sign-vector seed the codec uses unless a cache states another (the page
 * draws its vector once from a generator seeded with 42). */
#define TQ_DEFAULT_SIGN_SEED 42u

/* Human-readable name of a status. */
TQ_API const char *tq_status_string(tq_status status);

/* Bytes one token of one kv-head occupies in the planes:
 * d*k_bits/8 + 2*(d/32)*2 + d*v_bits/8 + (d/32)*2 (200 at k8v3, d=128; page
 * "Algorithm", its bytes-per-token-head figure).  Returns 0 for invalid parameters. */
TQ_API size_t tq_bytes_per_token_head(int32_t head_dim, int32_t k_bits, int32_t v_bits);

/* Size in bytes of each plane of `cache` (k_codes, k_scale, k_zero, v_codes,
 * v_scale) for its batch, heads and capacity; pointers are not read. */
TQ_API tq_status tq_plane_bytes(const tq_cache *cache, size_t out_bytes[5]);

/* The +-1 value sign vector the library applies for head_dim d and a seed
 * (host output, d int8 entries): entry i is -1 when the top bit of output i of
 * SplitMix64 started at `seed` is set (Steele, Lea & Flood, OOPSLA 2014),
 * else +1.  For one seed the d=64 vector is a prefix of the d=128 one, and so
 * on.  The page fixes one +-1 vector per head_dim, drawn once from a seeded
 * generator and hardcoded; here the seed is the cache's sign_seed (default
 * TQ_DEFAULT_SIGN_SEED = 42). */
TQ_API tq_status tq_sign_vector(int32_t head_dim, uint64_t seed, int8_t *host_out);

/* The Lloyd-Max tables for v_bits (host outputs): 2^v_bits centroids and
 * 2^v_bits - 1 boundaries (midpoints), fp32, ascending; the optimal quantizer
 * of a unit normal.  The page prints the 3-bit table (centroids +-0.24509,
 * +-0.75601, +-1.34391, +-2.15195; boundaries +-0.50055, +-1.04996, +-1.74793
 * and 0) and obtains the other widths by Lloyd-Max iteration on a unit normal. */
TQ_API tq_status tq_codebook(int32_t v_bits, float *host_centroids, float *host_boundaries);

/*
 * Append: quantise n_new tokens of K and V and write them into cache rows
 * [t0, t0 + n_new) of every (sequence, kv-head); no other row is written.
 * Page: updateAndFetch quantises just the tokens appended by the call.
 *  k, v      device bf16, element [b][h][t][j] at b*s[0] + h*s[1] + t*s[2] + j
 *            (strides in elements, head_dim contiguous); pointers 16-byte
 *            aligned and strides multiples of 8.
 *  t0        first row, 0 <= t0 and t0 + n_new <= capacity.
 * n_new = 0 is a no-op.
 */
TQ_API tq_status tq_encode_append(const tq_cache *cache, const void *k, const int64_t k_strides[3],
                           const void *v, const int64_t v_strides[3], int64_t t0, int64_t n_new,
                           tq_stream_t stream);

/*
 * Fetch: dequantise rows [t0, t0 + n) to K and V, [batch][H][n][d] contiguous,
 * bf16 (round to nearest even) or fp32 per out_dtype.  Either output may be
 * NULL to skip it.  Keys: (code + zero) * scale in fp32, the add first (page,
 * joint K/V decoder paragraph).  Values: signs * FWHT(centroid[code] * rms)
 * / sqrt(d) (the transform first, the sign multiply after it).  Outputs 32-byte aligned.
 */
TQ_API tq_status tq_decode(const tq_cache *cache, int64_t t0, int64_t n, tq_dtype out_dtype, void *k_out,
                    void *v_out, tq_stream_t stream);

/*
 * Deferred fetch: value rows [t0, t0 + n) still in the rotated domain,
 * centroid[code] * rms per element with no inverse transform and no signs,
 * [batch][H][n][d] contiguous, fp32 or bf16 (round to nearest even of the fp32
 * product).  Page section "Deferred inverse FWHT": attention is linear in the
 * values, so an attention kernel outside this library can form its weighted
 * sum on these rows and bring the result back once per query row with
 * tq_unrotate.  v_out 32-byte aligned.
 */
TQ_API tq_status tq_decode_values_rotated(const tq_cache *cache, int64_t t0, int64_t n, tq_dtype out_dtype,
                                          void *v_out, tq_stream_t stream);

/*
 * Un-rotation of vectors formed in the rotated domain: out = signs *
 * FWHT(x) / sqrt(d) for each of `rows` rows of head_dim elements (the second
 * half of the value dequantisation; page section "Deferred inverse FWHT"),
 * signs being tq_sign_vector(head_dim, sign_seed) -- the seed of the cache
 * the rows came from.
 *  x, out    device, [rows][head_dim] contiguous, fp32 or bf16 each
 *            (in_dtype, out_dtype); 32-byte aligned; out may equal x when the
 *            dtypes match (in place).
 * rows = 0 is a no-op.
 */
TQ_API tq_status tq_unrotate(int32_t head_dim, uint64_t sign_seed, tq_dtype in_dtype, const void *x, int64_t rows,
                             tq_dtype out_dtype, void *out, tq_stream_t stream);

/*
 * Cache lifecycle: copy token rows [src_t0, src_t0 + n) of every (sequence,
 * kv-head) of `src` into rows [dst_t0, dst_t0 + n) of `dst`, all five planes,
 * byte for byte.  Groups run along head_dim only, so token slices are
 * byte-safe (page section "Architecture in mlx-bun"); with it the caller
 * snapshots, restores and clones caches and grows capacity (copy into a
 * larger cache).  The two caches must agree in head_dim, bit widths, kv-heads,
 * batch and sign_seed (else TQ_ERR_SHAPE); capacities may differ.  Within one cache the ranges must not
 * overlap unless identical (then nothing moves).  n = 0 is a no-op.
 */
TQ_API tq_status tq_cache_copy_rows(const tq_cache *dst, int64_t dst_t0, const tq_cache *src, int64_t src_t0,
                                    int64_t n, tq_stream_t stream);

/*
 * Cache lifecycle: zero token rows [t0, t0 + n) of every (sequence, kv-head),
 * all planes.  Trimming a cache to length L is clearing [L, capacity): rows
 * appended there afterwards give the same bytes as in a cache that never held
 * the trimmed tokens.  n = 0 is a no-op.
 */
TQ_API tq_status tq_cache_clear_rows(const tq_cache *cache, int64_t t0, int64_t n, tq_stream_t stream);

/* Workspace bytes tq_decode_attention needs for these sizes (0 if invalid). */
TQ_API size_t tq_attention_workspace_bytes(const tq_cache *cache, int32_t q_heads, int64_t seq_len);

/*
 * Decode attention with dequantise-on-fetch, one query token per sequence:
 *   out[b][h] = sum_t softmax_t(q[b][h] . k_hat[b][h/G][t] * softmax_scale) v_hat[b][h/G][t]
 * over cache rows t in [0, seq_len), G = q_heads / num_kv_heads (GQA: q-head
 * h reads kv-head h / G).  Keys and values are dequantised inside the kernel;
 * values stay in the rotated domain and the output is un-rotated once per
 * (sequence, q-head) ("Deferred inverse FWHT").  Accumulation is fp32.
 *  q        device bf16 [batch][q_heads][d] contiguous, 16-byte aligned.
 *  out      device fp32 [batch][q_heads][d] contiguous, 16-byte aligned.
 *  workspace  device scratch of at least tq_attention_workspace_bytes(),
 *           16-byte aligned; its contents need no initialisation.
 * The token being generated must have been appended first (tq_encode_append
 * with t0 = seq_len - 1), as the page's updateAndFetch does.
 * Every head_dim, bit pair and group size G >= 1 is covered: head_dims 64,
 * 128 and 256 with 8- or 4-bit keys and 2-, 3- or 4-bit values run a
 * specialised kernel (blocks of 8 q-heads, one CTA per block, columns past G
 * dropped),
 * the rest a generic one (code widths read at run time, groups in blocks of
 * 8 q-heads); both meet the same tolerance.
 */
TQ_API tq_status tq_decode_attention(const tq_cache *cache, const void *q, int32_t q_heads, int64_t seq_len,
                              float softmax_scale, float *out, void *workspace, size_t workspace_bytes,
                              tq_stream_t stream);

/*
 * Decode attention without any device allocation -- the pages have no
 * counterpart to this entry point; it exists for callers that cannot obtain
 * scratch memory.  Same arguments, output and tolerance as tq_decode_attention
 * minus the workspace, for the specialised parameters only (head_dim 64, 128
 * or 256, 8- or 4-bit keys, 2-, 3- or 4-bit values, any group size; others
 * return TQ_ERR_UNSUPPORTED).  Typical callers: code running inside another
 * framework's memory manager that may not call cudaMalloc/cudaFree itself
 * (both can synchronise the device and fragment a pool someone else owns),
 * and plugin-style integrations with no allocator handle to pass a workspace
 * from.
 *  - Scratch: a fixed 16 MiB array inside the library, reserved on every GPU
 *    that loads the library for the life of the process.  The split count is
 *    reduced when needed so the partials fit; if even one split needs more
 *    than 16 MiB (batch * num_kv_heads * ceil(G/8) * 8 * (d+2) * 4 bytes,
 *    i.e. batch * num_kv_heads * ceil(G/8) > 7943, 4032 or 2032 at head_dim
 *    64, 128 or 256),
 *    the call returns TQ_ERR_SCRATCH and launches nothing.
 *  - The first call on each device looks up the array's device address (a
 *    runtime query, not an allocation); make that first call before any
 *    stream capture.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it needs to start at zero.  Calls whose kernels overlap on the
 *    GPU (different streams, or different host threads) race on it: order
 *    them.
 */
TQ_API tq_status tq_decode_attention_noalloc(const tq_cache *cache, const void *q, int32_t q_heads, int64_t seq_len,
                                             float softmax_scale, float *out, tq_stream_t stream);

/* Workspace bytes tq_multi_token_attention needs for these sizes (0 if invalid). */
TQ_API size_t tq_multi_token_workspace_bytes(const tq_cache *cache, int32_t q_heads, int64_t m_queries,
                                             int64_t seq_len);

/*
 * Causal attention for M query rows per sequence, the forward pass of a chunk
 * of M tokens appended together (the page's multi-token forward shapes are
 * M = 1, 4 and 128: "Packed-value decode fusion investigation"; chunked
 * prefill and speculative verification take the same form).  The chunk's own
 * rows are the cache's last M rows, appended first (tq_encode_append with
 * t0 = seq_len - M, n = M); query row i (0-based) sees rows
 * [0, seq_len - M + i], itself included and the later rows of the chunk not:
 *   out[b][i][h] = sum_{t <= seq_len-M+i} softmax_t(q[b][i][h] . k_hat[b][h/G][t]
 *                  * softmax_scale) v_hat[b][h/G][t]
 * Same dequantise-on-fetch method, deferred un-rotation, fp32 accumulation
 * and tolerance as tq_decode_attention, for every head_dim, bit pair and
 * group size; M = 1 gives decode attention.  The cache rows of one kv-head are
 * read once for up to 32 (query row, q-head) pairs at head_dim <= 128, 16 at
 * 256 and 8 at 512.
 *  q        device bf16 [batch][M][q_heads][d] contiguous, 16-byte aligned.
 *  out      device fp32 [batch][M][q_heads][d] contiguous, 16-byte aligned.
 *  workspace  device scratch of at least tq_multi_token_workspace_bytes(),
 *           16-byte aligned; its contents need no initialisation.
 * Errors: TQ_ERR_SHAPE if M < 1, M > seq_len, or batch * M * q_heads or
 * num_kv_heads * ceil(M * G / 8) is too large for one launch (2^30 rows,
 * 65535 column blocks); otherwise as tq_decode_attention.
 */
TQ_API tq_status tq_multi_token_attention(const tq_cache *cache, const void *q, int32_t q_heads, int64_t m_queries,
                                          int64_t seq_len, float softmax_scale, float *out, void *workspace,
                                          size_t workspace_bytes, tq_stream_t stream);

/* 1 if tq_decode_attention covers these parameters (every valid head_dim and
 * bit pair, group_size >= 1), else 0. */
TQ_API int tq_attention_supported(int32_t head_dim, int32_t k_bits, int32_t v_bits, int32_t group_size);

/*
 * Device-side error word.  Kernels that wait on asynchronous copies give up
 * after a bounded number of polls and record a non-zero code here instead of
 * hanging.  tq_device_error() synchronises the device, copies the word into
 * *host_code and clears it.
 */
TQ_API tq_status tq_device_error(uint32_t *host_code);

/* Code a bounded wait that gave up ORs into the device error word. */
#define TQ_DEVICE_ERR_WAIT_TIMEOUT 1u

/*
 * Failure-path check (no counterpart in the pages): launches one warp that
 * waits, through the same bounded wait every kernel of the library uses for
 * its asynchronous copies, on a shared-memory barrier that nothing will ever
 * complete.  The wait gives up after its limit (about 2 s of device time),
 * ORs TQ_DEVICE_ERR_WAIT_TIMEOUT into the device error word, and the kernel
 * returns.  It touches no memory outside its own shared memory and the error
 * word, and the context stays usable.  TQ_ERR_CUDA if the launch fails.
 */
TQ_API tq_status tq_check_wait_timeout(tq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
