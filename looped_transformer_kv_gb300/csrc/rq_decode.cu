// ResidualQuant split-KV decode attention over the packed cache, and the split combine.
//
// Scores and values are rebuilt inside attention (rit.work summary, "How each pass's KV
// cache is reconstructed"): for a loop-l query q and cached token t
//   score_t = a_t * (q . ref_hat_t) + (R q) . e_t,        e_t = deq(res_l,t)
//   out     = (sum_t p_t a_t ref_hat_t + R^T sum_t p_t e_t + p_pend v_pend) / sum p
// so the rotation touches the query once and the value accumulator once, and no
// decompressed K/V ever reaches memory.  The final loop is the reference itself (a = 1,
// no residual).
#include "rq_common.cuh"
#include "rq_kernels.h"

namespace rq {
namespace {

constexpr int kSplitChunk = 128;  // split boundaries: multiples of the kernels' tiles

// One warp per (b, query head, loop in the call): merge the split partials, add the
// current token's BF16 K/V, undo the rotation on the residual accumulator, store bf16.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const int8_t* __restrict__ v_signs,
                                                      const uint16_t* __restrict__ q,
                                                      const uint16_t* __restrict__ pending,
                                                      const float* __restrict__ ws,
                                                      const unsigned* __restrict__ err,
                                                      uint16_t* __restrict__ out, int B, int Hq,
                                                      int H, int loop_count, int n_splits,
                                                      float scale_log2) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = int64_t(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (wid >= int64_t(B) * Hq * loop_count) return;
  const int li = int(wid % loop_count);
  const int hq = int((wid / loop_count) % Hq);
  const int b = int(wid / (int64_t(loop_count) * Hq));
  const int h = hq / (Hq / H);
  const uint16_t* kpp = pending ? pending + ((int64_t(b) * 2 + 0) * loop_count + li) * H * D + int64_t(h) * D
                                : nullptr;
  const uint16_t* vpp = pending ? pending + ((int64_t(b) * 2 + 1) * loop_count + li) * H * D + int64_t(h) * D
                                : nullptr;
  combine_column<D>(ws + wid * n_splits * int64_t(partial_floats_d(D)), n_splits, q + wid * D, kpp, vpp,
                    v_signs ? v_signs + int64_t(h) * D : nullptr, scale_log2, err && *err,
                    out + wid * D, lane);
}

}  // namespace

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

SplitPlan plan_splits_for(const rq_shape& s, int max_ctx, int ctas_per_sm, int chunk) {
  SplitPlan p;
  const int64_t units = int64_t(s.batch) * s.n_kv_heads;
  const int64_t slots = int64_t(device_sm_count()) * (ctas_per_sm < 1 ? 1 : ctas_per_sm);
  const int tiles = max_ctx > 0 ? (max_ctx + chunk - 1) / chunk : 1;
  double best = 1e300;
  int best_per = tiles;
  for (int splits = 1; splits <= tiles && splits <= 256; ++splits) {
    const int per = (tiles + splits - 1) / splits;           // tiles per split
    const int real = (tiles + per - 1) / per;
    const int64_t waves = (units * real + slots - 1) / slots;
    const double cost = double(waves) * (per + 1.0);         // + one tile of set-up per split
    if (cost < best - 1e-9) {
      best = cost;
      best_per = per;
    }
  }
  p.tokens_per_split = best_per * chunk;
  p.n_splits = (tiles + best_per - 1) / best_per;
  return p;
}

SplitPlan plan_splits_bf16(const rq_shape& s, int max_ctx) {
  return plan_splits_for(s, max_ctx, 8, kSplitChunk);
}

SplitPlan plan_splits(const rq_shape& s, int loop_count, int max_ctx) {
  // the larger of the two kernels' plans over every loop range of this length
  SplitPlan best = plan_splits_bf16(s, max_ctx);
  for (int lb = 0; lb + loop_count <= s.n_loops; ++lb) {
    const SplitPlan p = plan_splits_rq(s, lb, loop_count, max_ctx);
    if (p.n_splits > best.n_splits) best = p;
  }
  return best;
}

size_t partial_floats(const rq_shape& s) { return partial_floats_d(s.head_dim); }

cudaError_t launch_rq_decode(const rq_shape& s, const rq_cache& cache, const rq_paging* paging,
                             const uint16_t* q,
                             int loop_begin, int loop_count, const uint16_t* pending,
                             const int32_t* ctx_lens, int max_ctx, uint16_t* out, float* ws,
                             cudaStream_t stream, const DecodeHooks* hooks) {
  const SplitPlan plan = plan_splits_rq(s, loop_begin, loop_count, max_ctx);
  unsigned* err = reinterpret_cast<unsigned*>(ws);
  const size_t tb = ws_ticket_bytes(s, loop_count);
  unsigned* tickets = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(ws) + kWsHeaderBytes);
  float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + kWsHeaderBytes + tb);
  cudaError_t e = cudaMemsetAsync(ws, 0, kWsHeaderBytes + tb, stream);   // error word, tickets
  if (e != cudaSuccess) return e;
  const bool in_kernel = decode_combines_in_kernel(s, loop_begin, loop_count);
  e = launch_rq_decode_mma(s, cache, paging, q, loop_begin, loop_count, ctx_lens, plan.n_splits,
                           plan.tokens_per_split, pending, out, part, in_kernel ? tickets : nullptr,
                           err, stream, hooks);
  if (e != cudaSuccess) return e;
  if (in_kernel) return cudaSuccess;
  return launch_combine(s, cache.rot_signs[1], q, loop_count, pending, plan.n_splits, out, part,
                        err, stream);
}

cudaError_t launch_combine(const rq_shape& s, const int8_t* v_signs, const uint16_t* q,
                           int loop_count, const uint16_t* pending, int n_splits,
                           uint16_t* out, const float* part, const unsigned* err,
                           cudaStream_t stream) {
  const int64_t warps = int64_t(s.batch) * s.n_q_heads * loop_count;
  const unsigned blocks = unsigned((warps + 3) / 4);
  const float scale = s.softmax_scale > 0.f ? s.softmax_scale : 1.0f / sqrtf(float(s.head_dim));
  if (s.head_dim == 128)
    combine_kernel<128><<<blocks, 128, 0, stream>>>(v_signs, q, pending, part, err, out, s.batch,
                                                    s.n_q_heads, s.n_kv_heads, loop_count,
                                                    n_splits, scale * kLog2e);
  else
    combine_kernel<64><<<blocks, 128, 0, stream>>>(v_signs, q, pending, part, err, out, s.batch,
                                                   s.n_q_heads, s.n_kv_heads, loop_count,
                                                   n_splits, scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace rq
