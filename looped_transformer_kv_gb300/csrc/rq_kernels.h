// Internal launchers behind the C ABI (host code; no validation here).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rq.h"

namespace rq {

struct SplitPlan {
  int n_splits;          // split-KV partitions of the context
  int tokens_per_split;  // multiple of the kernel's token chunk
};

SplitPlan plan_splits(const rq_shape& s, int loop_count, int max_ctx);
size_t partial_floats(const rq_shape& s);  // floats of one partial record

cudaError_t launch_encode(const rq_shape& s, const rq_cache& cache, const uint16_t* kv_new,
                          const int64_t strides[5], const int32_t* positions, int32_t pos_begin,
                          int32_t n_new, cudaStream_t stream);

cudaError_t launch_rq_decode(const rq_shape& s, const rq_cache& cache, const uint16_t* q,
                             int loop_begin, int loop_count, const uint16_t* pending,
                             const int32_t* ctx_lens, int max_ctx, uint16_t* out, float* ws,
                             cudaStream_t stream);

cudaError_t launch_bf16_decode(const rq_shape& s, const uint16_t* k, const uint16_t* v,
                               const uint16_t* q, int loop_begin, int loop_count,
                               const uint16_t* pending, const int32_t* ctx_lens, int max_ctx,
                               uint16_t* out, float* ws, cudaStream_t stream);

cudaError_t launch_combine(const rq_shape& s, const int8_t* v_signs, const uint16_t* q,
                           int loop_count, const uint16_t* pending, int n_splits,
                           uint16_t* out, const float* ws, cudaStream_t stream);

int device_sm_count();

}  // namespace rq
