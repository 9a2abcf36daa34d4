/*
 * librq test hooks: entry points that exist only so that the test suite can drive failure
 * paths without faulting, trapping or hanging a GPU.  No product call uses them.
 */
#ifndef RQ_TEST_H_
#define RQ_TEST_H_

#include "rq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* rq_decode_attention (same arguments, same validation, same workspace) with the copy of the
 * first 64-token tile of every split withheld and the pipeline wait limit set to
 * wait_limit_ns (in (0, 2e9]; product calls use 2 s).  The wait for that tile can only run
 * out -- nothing is in flight for it -- so every split with cached tokens takes the
 * bounded-wait failure path: it sets the workspace error word, waits (bounded again) for its
 * other copies, which complete normally, and leaves its outputs NaN.  Each such split takes
 * about twice wait_limit_ns.  The CUDA context stays usable afterwards.  (The method's pages
 * have no counterpart: this is a test of the library's own error handling.) */
rq_status rq_test_decode_attention_wait_runs_out(const rq_shape* shape, const rq_cache* cache,
                                                 const uint16_t* q, int32_t loop_begin,
                                                 int32_t loop_count, const uint16_t* pending_kv,
                                                 const int32_t* ctx_lens, int32_t max_ctx,
                                                 uint16_t* out, void* ws, size_t ws_bytes,
                                                 uint64_t wait_limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RQ_TEST_H_ */
