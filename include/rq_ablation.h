/*
 * librq ablation rows: the method with one of its steps changed, for measuring what each
 * step buys in error, bytes and time ("ResidualQuant: KV Cache Quantization for Looped
 * Transformers with 2-Bit Residuals", abstract; rit.work summary, "When ResidualQuant changes
 * the infrastructure plan": the ablation ladder from direct INT2 through the reference, the
 * least-squares scale and the rotation to loop-wise mixed precision).  Same cache layout,
 * shapes and conventions as rq.h.
 */
#ifndef RQ_ABLATION_H_
#define RQ_ABLATION_H_

#include "rq.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RQ_ALPHA_LEAST_SQUARES = 0, /* the method: a_l = <x_l, ref_hat> / <ref_hat, ref_hat>       */
  RQ_ALPHA_ONE = 1,           /* a_l = 1: residual against the unscaled reference            */
  RQ_ALPHA_ZERO = 2           /* a_l = 0: the residual array holds the loop's own state,
                                 rotated and quantised directly (no reference part)          */
} rq_alpha_mode;

/* rq_encode_append with a_l fixed by alpha_mode (stored as such in the alpha arrays; the
 * final loop is the INT4 reference in every mode).  Same arguments and validation otherwise;
 * an alpha_mode outside the enum returns RQ_ERR_INVALID_ARG. */
rq_status rq_ablation_encode_append(const rq_shape* shape, const rq_cache* cache,
                                    const uint16_t* kv_new, const int64_t strides[5],
                                    const int32_t* positions, int32_t pos_begin, int32_t n_new,
                                    int32_t alpha_mode, void* stream);

/* Causal per-loop decode attention of residual loop `loop` (0 <= loop < L-1) over a cache
 * encoded with RQ_ALPHA_ONE (mode 1: the a arrays are not read, a = 1) or RQ_ALPHA_ZERO
 * (mode 2: neither the reference nor the a arrays are read; the score and the value are the
 * loop's own rotated codes).  Arguments as rq_decode_attention with loop_begin = loop and
 * loop_count = 1, the same workspace size; supported shapes: one query head per kv-head and
 * head dim 128 (RQ_ERR_UNSUPPORTED otherwise).  The final loop is decoded by
 * rq_decode_attention in every mode. */
rq_status rq_ablation_decode_attention(const rq_shape* shape, const rq_cache* cache, int32_t mode,
                                       const uint16_t* q, int32_t loop, const uint16_t* pending_kv,
                                       const int32_t* ctx_lens, int32_t max_ctx, uint16_t* out,
                                       void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RQ_ABLATION_H_ */
