// rq_decode_attention_noalloc: decode attention for callers that cannot allocate device
// memory.  The split-KV scratch (error word, split tickets, partial records) lives in one
// file-scope device array instead of a caller-provided workspace.
#include <mutex>

#include "rq_common.cuh"
#include "rq_kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB, fixed at build time

// Held by every GPU that loads the library, from load until process exit.
static __device__ __align__(256) unsigned char g_rq_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];   // device address of the array per device, once found

// Device address of the scratch array on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is looked up with that device current.
// Only a successful lookup is kept: a failed one (for example a first call made during
// stream capture) is retried by the next call, and its error is cleared so that it does not
// surface in a later, unrelated cudaGetLastError.
rq_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return RQ_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_rq_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return RQ_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return RQ_OK;
}

}  // namespace

extern "C" size_t rq_decode_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" rq_status rq_decode_attention_noalloc(const rq_shape* shape, const rq_cache* cache,
                                                 const uint16_t* q, int32_t loop_begin,
                                                 int32_t loop_count, const uint16_t* pending_kv,
                                                 const int32_t* ctx_lens, int32_t max_ctx,
                                                 uint16_t* out, void* stream) {
  // the same checks, in the same order, as rq_decode_attention: same status for same arguments
  const rq_status valid =
      rq::validate_decode(shape, cache, q, loop_begin, loop_count, ctx_lens, max_ctx, out);
  if (valid != RQ_OK) return valid;
  // a valid call whose split-KV scratch would not fit the array: refused, nothing enqueued
  if (rq_decode_workspace_bytes(shape, loop_count, max_ctx) > kNoAllocScratchBytes)
    return RQ_ERR_WORKSPACE;
  void* ws = nullptr;
  const rq_status st = scratch_for_current_device(&ws);
  if (st != RQ_OK) return st;
  // the scratch array's error word and tickets are cleared by the call itself; every partial
  // record the combine reads is rewritten by the split kernels, so nothing else needs clearing
  return rq_decode_attention(shape, cache, q, loop_begin, loop_count, pending_kv, ctx_lens,
                             max_ctx, out, ws, kNoAllocScratchBytes, stream);
}
