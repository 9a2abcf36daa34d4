/*
 * librq synthetic inputs: the seeded generator of looped K/V states and queries, on the
 * GPU.  Not part of ResidualQuant itself (the pages have no counterpart); it writes
 * benchmark and test inputs straight into device memory.
 *
 * Every value is a function of (seed, field, coordinates): Philox4x32-10 (Salmon et al.,
 * "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11) with counter
 *   c0 = token position (queries: decode step), c1 = batch index,
 *   c2 = head << 16 | kv << 15 | loop << 8 | channel, c3 = field << 24 | layer << 8 | sub,
 * key = (seed low 32 bits, seed high 32 bits), followed by IEEE fp32 operations that are
 * correctly rounded (no contraction), then round-to-nearest-even to bf16.  The host-side
 * twin (numpy) produces bit-identical values.
 *   normal  z  = (sum of the twelve 10-bit fields of one Philox block - 6138) / 1024
 *   base       = z (field 1, sub 0); Student-t(3): z0 / sqrt(max(((z1^2 + z2^2) + z3^2)/3, 2^-10))
 *                with z0..z3 drawn with sub 0..3; times outlier_mult on outlier channels
 *   u_l        = 0.8 + 0.4 * ((word0 >> 8) + 0.5) * 2^-24       (field 3, channel 0)
 *   x          = bf16(u_l * base + sigma_l * n),  n normal (field 2)
 *   query      = bf16(z) (field 4, c0 = step, head = query head, kv = 0)
 */
#ifndef RQ_SYNTH_H_
#define RQ_SYNTH_H_

#include <stddef.h>
#include <stdint.h>

#include "rq.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  uint64_t seed;
  int32_t layer;          /* 0..65535                                           */
  int32_t head_dim;       /* d <= 256                                          */
  int32_t n_kv_heads;
  int32_t dist;           /* 0: normal base, 1: Student-t with 3 dof            */
  float sigma[RQ_MAX_LOOPS]; /* inter-loop noise of each loop (fp32 values)     */
  float outlier_mult;
  int32_t n_outliers;     /* outlier channels per (kv-head, K/V), 0..8          */
  const int32_t* outlier_table; /* device int32 [Hkv][2][max(n_outliers,1)]      */
} rq_synth_params;

/* States for batch b in [b0, b0+nb), token t in [t0, t0+nt), kv in {0, 1},
 * loop l in [l0, l0+nl), every kv-head h and channel i, written as bf16 at
 *   out + (b-b0)*strides[0] + (t-t0)*strides[1] + kv*strides[2] + (l-l0)*strides[3]
 *       + h*strides[4] + i          (strides in elements). */
rq_status rq_synth_states(const rq_synth_params* p, uint16_t* out, const int64_t strides[5],
                          int32_t b0, int32_t nb, int32_t t0, int32_t nt, int32_t l0,
                          int32_t nl, void* stream);

/* Queries bf16 [nb][n_q_heads][nl][d] for batch b0.., loops l0.., decode step `step`. */
rq_status rq_synth_queries(const rq_synth_params* p, uint16_t* out, int32_t n_q_heads,
                           int32_t b0, int32_t nb, int32_t l0, int32_t nl, int32_t step,
                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RQ_SYNTH_H_ */
