// C ABI of librq: argument validation, then the internal launchers.  Nothing is
// enqueued unless every check passes; no exception crosses this boundary.
#include <cmath>
#include <new>

#include "../../include/rq_ablation.h"
#include "../../include/rq_test.h"
#include "rq_common.cuh"
#include "rq_kernels.h"

namespace {

__global__ void advance_ctx_kernel(int32_t* ctx_lens, int32_t batch, int32_t n, int32_t cap) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) {
    const int64_t v = int64_t(ctx_lens[b]) + n;
    ctx_lens[b] = int32_t(v > cap ? cap : v);
  }
}

rq_status check_shape(const rq_shape* s) {
  if (!s) return RQ_ERR_INVALID_ARG;
  if (s->batch <= 0 || s->n_q_heads <= 0 || s->n_kv_heads <= 0 || s->capacity <= 0 ||
      s->n_loops <= 0)
    return RQ_ERR_INVALID_ARG;
  if (s->n_q_heads % s->n_kv_heads != 0) return RQ_ERR_INVALID_ARG;
  if (s->capacity % 64 != 0) return RQ_ERR_INVALID_ARG;
  if (s->group != 32) return RQ_ERR_UNSUPPORTED;
  if (s->head_dim != 64 && s->head_dim != 128) return RQ_ERR_UNSUPPORTED;
  if (s->n_loops > RQ_MAX_LOOPS) return RQ_ERR_UNSUPPORTED;
  if (s->batch > 65535 || s->n_kv_heads > 65535) return RQ_ERR_UNSUPPORTED;
  for (int l = 0; l < s->n_loops - 1; ++l)
    if (s->res_bits[l] != 2 && s->res_bits[l] != 4) return RQ_ERR_UNSUPPORTED;
  if (!(s->softmax_scale >= 0.f) || std::isinf(s->softmax_scale)) return RQ_ERR_INVALID_ARG;
  return RQ_OK;
}

rq_status check_cache(const rq_shape* s, const rq_cache* c) {
  (void)s;
  if (!c || !c->data || !c->rot_signs[0] || !c->rot_signs[1]) return RQ_ERR_INVALID_ARG;
  // every piece of a record a stage copies starts at a multiple of 128 bytes of its record,
  // and records are a multiple of 128 bytes long: 16-byte alignment of the base suffices
  if ((reinterpret_cast<uintptr_t>(c->data) & 15) != 0) return RQ_ERR_INVALID_ARG;
  return RQ_OK;
}

// Decode arguments other than the workspace.
rq_status check_decode_args(const rq_shape* s, const uint16_t* q, int32_t loop_begin,
                            int32_t loop_count, const int32_t* ctx_lens, int32_t max_ctx,
                            uint16_t* out) {
  if (!q || !ctx_lens || !out) return RQ_ERR_INVALID_ARG;
  if (loop_count < 1 || loop_begin < 0 || loop_begin + loop_count > s->n_loops)
    return RQ_ERR_INVALID_ARG;
  if (max_ctx < 0 || max_ctx > s->capacity) return RQ_ERR_INVALID_ARG;
  if (int64_t(s->batch) * s->n_q_heads * loop_count > (int64_t(1) << 31))
    return RQ_ERR_UNSUPPORTED;
  return RQ_OK;
}

rq_status check_decode(const rq_shape* s, const uint16_t* q, int32_t loop_begin,
                       int32_t loop_count, const int32_t* ctx_lens, int32_t max_ctx,
                       uint16_t* out, void* ws, size_t ws_bytes) {
  const rq_status st = check_decode_args(s, q, loop_begin, loop_count, ctx_lens, max_ctx, out);
  if (st != RQ_OK) return st;
  const size_t need = rq_decode_workspace_bytes(s, loop_count, max_ctx);
  if (!ws || ws_bytes < need) return RQ_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return RQ_ERR_WORKSPACE;
  return RQ_OK;
}

rq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA; }

rq_status check_paging(const rq_shape* s, const rq_paging* pg) {
  if (!pg || !pg->block_table || pg->max_pages <= 0 || pg->n_pages <= 0)
    return RQ_ERR_INVALID_ARG;
  if (int64_t(s->capacity) != int64_t(64) * pg->max_pages) return RQ_ERR_INVALID_ARG;
  if (int64_t(pg->n_pages) * s->n_kv_heads * 64 > (int64_t(1) << 40)) return RQ_ERR_UNSUPPORTED;
  return RQ_OK;
}

// Bytes of one token of one kv-head, K and V, every array of the packed cache.
size_t token_head_bytes(const rq_shape* s) {
  const size_t d = size_t(s->head_dim), ng = d / 32;
  size_t per = d / 2 + 4 * ng;
  for (int l = 0; l < s->n_loops - 1; ++l) per += d * size_t(s->res_bits[l]) / 8 + 4 * ng + 2;
  return 2 * per;
}

rq_status encode_common(const rq_shape* shape, const rq_cache* cache, const rq_paging* paging,
                        const uint16_t* kv_new, const int64_t strides[5],
                        const int32_t* positions, int32_t pos_begin, int32_t n_new,
                        void* stream, int alpha_mode = 0) {
  rq_status st = check_shape(shape);
  if (st != RQ_OK) return st;
  if ((st = check_cache(shape, cache)) != RQ_OK) return st;
  if (paging && (st = check_paging(shape, paging)) != RQ_OK) return st;
  if (!kv_new || !strides || n_new < 0) return RQ_ERR_INVALID_ARG;
  for (int k = 0; k < 5; ++k)
    if (strides[k] < 0) return RQ_ERR_INVALID_ARG;
  if (!positions && (pos_begin < 0 || int64_t(pos_begin) + n_new > shape->capacity))
    return RQ_ERR_INVALID_ARG;
  if (n_new == 0) return RQ_OK;
  try {
    return from_cuda(rq::launch_encode(*shape, *cache, paging, kv_new, strides, positions,
                                       pos_begin, n_new, static_cast<cudaStream_t>(stream),
                                       alpha_mode));
  } catch (...) {
    return RQ_ERR_INTERNAL;
  }
}

rq_status decode_common(const rq_shape* shape, const rq_cache* cache, const rq_paging* paging,
                        const uint16_t* q, int32_t loop_begin, int32_t loop_count,
                        const uint16_t* pending_kv, const int32_t* ctx_lens, int32_t max_ctx,
                        uint16_t* out, void* ws, size_t ws_bytes, void* stream,
                        const rq::DecodeHooks* hooks = nullptr) {
  rq_status st = check_shape(shape);
  if (st != RQ_OK) return st;
  if ((st = check_cache(shape, cache)) != RQ_OK) return st;
  if (paging && (st = check_paging(shape, paging)) != RQ_OK) return st;
  if ((st = check_decode(shape, q, loop_begin, loop_count, ctx_lens, max_ctx, out, ws,
                         ws_bytes)) != RQ_OK)
    return st;
  try {
    return from_cuda(rq::launch_rq_decode(*shape, *cache, paging, q, loop_begin, loop_count,
                                          pending_kv, ctx_lens, max_ctx, out,
                                          static_cast<float*>(ws),
                                          static_cast<cudaStream_t>(stream), hooks));
  } catch (...) {
    return RQ_ERR_INTERNAL;
  }
}

}  // namespace

namespace rq {

// Every check rq_decode_attention makes before its workspace check, in the same order, so
// that an entry point with its own scratch returns the same status for the same arguments.
rq_status validate_decode(const rq_shape* shape, const rq_cache* cache, const uint16_t* q,
                          int32_t loop_begin, int32_t loop_count, const int32_t* ctx_lens,
                          int32_t max_ctx, uint16_t* out) {
  rq_status st = check_shape(shape);
  if (st != RQ_OK) return st;
  if ((st = check_cache(shape, cache)) != RQ_OK) return st;
  return check_decode_args(shape, q, loop_begin, loop_count, ctx_lens, max_ctx, out);
}

}  // namespace rq

extern "C" {

size_t rq_cache_bytes(const rq_shape* s) {
  if (check_shape(s) != RQ_OK) return 0;
  return token_head_bytes(s) * size_t(s->capacity) * size_t(s->n_kv_heads) * size_t(s->batch);
}

size_t rq_record_bytes(const rq_shape* s) {
  if (check_shape(s) != RQ_OK) return 0;
  return size_t(rq::record_bytes(*s));
}

size_t rq_paged_cache_bytes(const rq_shape* s, int32_t n_pages) {
  if (check_shape(s) != RQ_OK || n_pages <= 0) return 0;
  return token_head_bytes(s) * 64 * size_t(n_pages) * size_t(s->n_kv_heads);
}

rq_status rq_encode_append(const rq_shape* shape, const rq_cache* cache, const uint16_t* kv_new,
                           const int64_t strides[5], const int32_t* positions, int32_t pos_begin,
                           int32_t n_new, void* stream) {
  return encode_common(shape, cache, nullptr, kv_new, strides, positions, pos_begin, n_new,
                       stream);
}

rq_status rq_paged_encode_append(const rq_shape* shape, const rq_cache* cache,
                                 const rq_paging* paging, const uint16_t* kv_new,
                                 const int64_t strides[5], const int32_t* positions,
                                 int32_t pos_begin, int32_t n_new, void* stream) {
  if (!paging) return RQ_ERR_INVALID_ARG;
  return encode_common(shape, cache, paging, kv_new, strides, positions, pos_begin, n_new,
                       stream);
}

size_t rq_decode_workspace_bytes(const rq_shape* s, int32_t loop_count, int32_t max_ctx) {
  if (check_shape(s) != RQ_OK || loop_count < 1 || max_ctx < 0) return 0;
  const rq::SplitPlan p = rq::plan_splits(*s, loop_count, max_ctx);
  return size_t(rq::kWsHeaderBytes) + rq::ws_ticket_bytes(*s, loop_count) +
         size_t(s->batch) * s->n_q_heads * loop_count * p.n_splits * rq::partial_floats(*s) *
             sizeof(float);
}

rq_status rq_decode_attention(const rq_shape* shape, const rq_cache* cache, const uint16_t* q,
                              int32_t loop_begin, int32_t loop_count, const uint16_t* pending_kv,
                              const int32_t* ctx_lens, int32_t max_ctx, uint16_t* out, void* ws,
                              size_t ws_bytes, void* stream) {
  return decode_common(shape, cache, nullptr, q, loop_begin, loop_count, pending_kv, ctx_lens,
                       max_ctx, out, ws, ws_bytes, stream);
}

rq_status rq_paged_decode_attention(const rq_shape* shape, const rq_cache* cache,
                                    const rq_paging* paging, const uint16_t* q,
                                    int32_t loop_begin, int32_t loop_count,
                                    const uint16_t* pending_kv, const int32_t* ctx_lens,
                                    int32_t max_ctx, uint16_t* out, void* ws, size_t ws_bytes,
                                    void* stream) {
  if (!paging) return RQ_ERR_INVALID_ARG;
  return decode_common(shape, cache, paging, q, loop_begin, loop_count, pending_kv, ctx_lens,
                       max_ctx, out, ws, ws_bytes, stream);
}

rq_status rq_bf16_decode_attention(const rq_shape* shape, const uint16_t* k, const uint16_t* v,
                                   const uint16_t* q, int32_t loop_begin, int32_t loop_count,
                                   const uint16_t* pending_kv, const int32_t* ctx_lens,
                                   int32_t max_ctx, uint16_t* out, void* ws, size_t ws_bytes,
                                   void* stream) {
  rq_status st = check_shape(shape);
  if (st != RQ_OK) return st;
  if (!k || !v) return RQ_ERR_INVALID_ARG;
  if (shape->n_q_heads / shape->n_kv_heads > 8) return RQ_ERR_UNSUPPORTED;
  if ((st = check_decode(shape, q, loop_begin, loop_count, ctx_lens, max_ctx, out, ws,
                         ws_bytes)) != RQ_OK)
    return st;
  try {
    return from_cuda(rq::launch_bf16_decode(*shape, k, v, q, loop_begin, loop_count, pending_kv,
                                            ctx_lens, max_ctx, out, static_cast<float*>(ws),
                                            static_cast<cudaStream_t>(stream)));
  } catch (...) {
    return RQ_ERR_INTERNAL;
  }
}

rq_status rq_test_decode_attention_wait_runs_out(const rq_shape* shape, const rq_cache* cache,
                                                 const uint16_t* q, int32_t loop_begin,
                                                 int32_t loop_count, const uint16_t* pending_kv,
                                                 const int32_t* ctx_lens, int32_t max_ctx,
                                                 uint16_t* out, void* ws, size_t ws_bytes,
                                                 uint64_t wait_limit_ns, void* stream) {
  if (wait_limit_ns == 0 || wait_limit_ns > 2000000000ull) return RQ_ERR_INVALID_ARG;
  const rq::DecodeHooks hooks{wait_limit_ns, true};
  return decode_common(shape, cache, nullptr, q, loop_begin, loop_count, pending_kv, ctx_lens,
                       max_ctx, out, ws, ws_bytes, stream, &hooks);
}

rq_status rq_ablation_encode_append(const rq_shape* shape, const rq_cache* cache,
                                    const uint16_t* kv_new, const int64_t strides[5],
                                    const int32_t* positions, int32_t pos_begin, int32_t n_new,
                                    int32_t alpha_mode, void* stream) {
  if (alpha_mode < RQ_ALPHA_LEAST_SQUARES || alpha_mode > RQ_ALPHA_ZERO) return RQ_ERR_INVALID_ARG;
  return encode_common(shape, cache, nullptr, kv_new, strides, positions, pos_begin, n_new,
                       stream, alpha_mode);
}

rq_status rq_ablation_decode_attention(const rq_shape* shape, const rq_cache* cache, int32_t mode,
                                       const uint16_t* q, int32_t loop, const uint16_t* pending_kv,
                                       const int32_t* ctx_lens, int32_t max_ctx, uint16_t* out,
                                       void* ws, size_t ws_bytes, void* stream) {
  rq_status st = check_shape(shape);
  if (st != RQ_OK) return st;
  if ((st = check_cache(shape, cache)) != RQ_OK) return st;
  if (mode != RQ_ALPHA_ONE && mode != RQ_ALPHA_ZERO) return RQ_ERR_INVALID_ARG;
  if (loop < 0 || loop >= shape->n_loops - 1) return RQ_ERR_INVALID_ARG;
  if ((st = check_decode(shape, q, loop, 1, ctx_lens, max_ctx, out, ws, ws_bytes)) != RQ_OK)
    return st;
  if (shape->n_q_heads != shape->n_kv_heads || shape->head_dim != 128) return RQ_ERR_UNSUPPORTED;
  try {
    return from_cuda(rq::launch_rq_ablation_decode(*shape, *cache, mode, q, loop, pending_kv,
                                                   ctx_lens, max_ctx, out, static_cast<float*>(ws),
                                                   static_cast<cudaStream_t>(stream)));
  } catch (...) {
    return RQ_ERR_INTERNAL;
  }
}

rq_status rq_advance_ctx(int32_t* ctx_lens, int32_t batch, int32_t n, int32_t capacity,
                         void* stream) {
  if (!ctx_lens || batch <= 0 || n < 0 || capacity <= 0) return RQ_ERR_INVALID_ARG;
  advance_ctx_kernel<<<(batch + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      ctx_lens, batch, n, capacity);
  return from_cuda(cudaGetLastError());
}

const char* rq_status_str(rq_status s) {
  switch (s) {
    case RQ_OK: return "RQ_OK";
    case RQ_ERR_INVALID_ARG: return "RQ_ERR_INVALID_ARG";
    case RQ_ERR_UNSUPPORTED: return "RQ_ERR_UNSUPPORTED";
    case RQ_ERR_WORKSPACE: return "RQ_ERR_WORKSPACE";
    case RQ_ERR_CUDA: return "RQ_ERR_CUDA";
    case RQ_ERR_INTERNAL: return "RQ_ERR_INTERNAL";
  }
  return "RQ_ERR_UNKNOWN";
}

}  // extern "C"
