/* synth.h -- seeded synthetic KV inputs, shared by the tests, the oracle
 * checks and the benchmark.  Holds none of the codec's arithmetic.
 *
 * Every value is a pure function of (stream seed, element counter), so any
 * row can be regenerated on its own.  Definitions:
 *   u64(s, i)     = output i of SplitMix64 started at s (Steele, Lea & Flood 2014)
 *   uniform(s, i) = ((u64(s, i) >> 11) + 0.5) * 2^-53                in (0, 1)
 *   normal(s, i)  = sqrt(-2 ln uniform(s, 2i)) * cos(2 pi uniform(s, 2i+1))   (Box-Muller)
 *   t5(s, i)      = normal(s, 6i) / sqrt(sum_{k=1..5} normal(s, 6i+k)^2 / 5) * sqrt(3/5)
 *                   (Student-t, 5 degrees of freedom, scaled to unit variance)
 * Streams of a workload with data seed S: K = u64(S,0), V = u64(S,1),
 * key channel scales = u64(S,2), queries = u64(S,3).
 * Element counter of K/V[b][h][t][j] (t = absolute token position):
 *   ((b*H + h) * 2^32 + t) * d + j
 * Key channel scale of (h, j): exp(sigma * normal(scale stream, h*d + j)),
 * one per (kv-head, channel), shared across batch and tokens.
 * Query counter of q[step][b][qh][j]: ((step*B + b)*QH + qh)*d + j.
 * Values are rounded to fp32 (nearest) and then to bf16 (nearest even).
 */
#ifndef TQ_SYNTH_H
#define TQ_SYNTH_H
#include <stdint.h>

#define TQS_V_NORMAL 0
#define TQS_V_T5 1

#ifdef __cplusplus
extern "C" {
#endif
/* Host: K, V bf16 bits, [B][H][n][d] contiguous, tokens [t_begin, t_begin+n) of
 * sequences [b_offset, b_offset+B). */
void tqs_host_kv(uint64_t data_seed, int B, int H, int d, int64_t t_begin, int64_t n, int b_offset,
                 double k_log_sigma, int v_dist, uint16_t *k_out, uint16_t *v_out);
/* Host: queries of one step, bf16 bits [B][QH][d]. */
void tqs_host_q(uint64_t data_seed, int64_t step, int B, int QH, int d, uint16_t *q_out);
uint64_t tqs_splitmix64(uint64_t seed, uint64_t i);
double tqs_normal(uint64_t stream, uint64_t i);
double tqs_t5(uint64_t stream, uint64_t i);
#ifdef __cplusplus
}
#endif
#endif
