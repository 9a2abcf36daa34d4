// Internal launchers behind the C ABI (host code; no validation here).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rq.h"

namespace rq {

constexpr int kMaxResPerBlock = 8;   // residual loops handled by one decode launch
constexpr int kTile = 64;            // tokens per tile record (and per decode stage)

// Tile record of the packed cache (include/rq.h): 64-row sections, the reference section
// (K codes, K meta, V codes, V meta) first, then one section per non-final loop (K codes,
// K meta, K a, V codes, V meta, V a).  Byte sizes and offsets; every one a multiple of 128.
__host__ __device__ inline int ref_section_bytes(int D) { return kTile * (D + 8 * (D / 32)); }
__host__ __device__ inline int loop_section_bytes(int D, int bits) {
  return kTile * (2 * (D * bits / 8) + 8 * (D / 32) + 4);
}
__host__ __device__ inline int loop_section_offset(int D, const int8_t* res_bits, int l) {
  int o = ref_section_bytes(D);
  for (int k = 0; k < l; ++k) o += loop_section_bytes(D, res_bits[k]);
  return o;
}
inline int64_t record_bytes(const rq_shape& s) {
  return loop_section_offset(s.head_dim, s.res_bits, s.n_loops - 1);
}
constexpr int kWsHeaderBytes = 256;  // workspace header: uint32 error word, then padding

// Variants of the decode kernel that keep, per residual loop, the rotated-query fragments
// masked to the loop's columns (4- or 8-column packing, 2-bit residual loops, residual-loop
// count fixed at compile time and >= 2): bytes of that region, else 0 (a lane's fragment is
// 8 bytes with the 4-column packing, 16 -- high and low parts -- with 8 columns).  Kernel and
// host use this one rule.
__host__ __device__ inline int masked_fragment_bytes(int D, bool res4, int nr, int pk) {
  const bool fixed = (D == 128 && (nr == 2 || nr == 3)) || (D == 64 && nr == 3);
  return ((pk == 1 || pk == 0) && !res4 && fixed) ? nr * (D / 32) * 2 * 32 * (pk == 0 ? 16 : 8) : 0;
}

// Packed-cache decode workspace: header, then one uint32 ticket per (sequence, kv-head, query
// block) counting the splits that have stored their partial records (the last one combines),
// then the partial records.  Header and tickets are cleared by every call.
inline size_t ws_ticket_bytes(const rq_shape& s, int loop_count) {
  // blocks per kv-head <= query heads per kv-head x loops in the call
  const size_t n = size_t(s.batch) * s.n_q_heads * (loop_count > 0 ? loop_count : 1);
  return (n * 4 + 255) / 256 * 256;
}

// A block of query columns handled by one launch: query heads [gi0, gi0 + gw) of each
// kv-head (gw a power of two <= 8) for loops [lb, lb + nl); residual loops [r0, r0 + nr).
struct QueryBlock {
  int gi0, gw, lb, nl, r0, nr;
};

// Shared-memory layout of the tensor-core decode kernel (byte offsets).  The stage region
// also holds the four warps' partial accumulators when the tiles are done.
struct SmemLayout {
  int qf, qr2, qr4, qrm, qsum, qrsum, ob, red, cnt, pg, bars, total;
};

// page_ids: physical page ids of a split's tiles kept for a paged cache (0 otherwise);
// qrm_bytes: the rotated-query fragments masked per residual loop (0 if the variant keeps
// none).
__host__ __device__ inline SmemLayout smem_layout(int D, bool res4, int stages, int stage_bytes,
                                                  int page_ids, int qrm_bytes) {
  const int NG = D / 32, NQ = 8, W = 4;
  SmemLayout s;
  int o = stages * stage_bytes;
  const int merge = W * NQ * (2 * D + 4) * 4;
  if (o < merge) o = merge;
  o = (o + 15) & ~15;
  const int frag = NG * 2 * 32 * 16;   // hi and lo f16x2 pairs per lane
  s.qf = o;    o += frag;
  s.qr2 = o;   o += frag;
  s.qr4 = o;   o += res4 ? frag : 0;
  s.qrm = o;   o += qrm_bytes;
  s.qsum = o;  o += NG * NQ * 4;
  s.qrsum = o; o += NG * NQ * 4;
  s.ob = o;    o += 8 * 32 * 4;       // B fragments of the score offset MMAs
  s.red = o;   o += 2 * W * NQ * 4;
  s.cnt = o;   o += 16 * 4;           // stage release counters, tiles issued
  s.pg = o;    o += page_ids * 4;
  o = (o + 7) & ~7;
  s.bars = o;  o += stages * 8;
  s.total = o;
  return s;
}

// Split partial record: m, l, two pad floats, acc_ref[D], acc_res[D] (16-byte aligned rows).
__host__ __device__ constexpr size_t partial_floats_d(int D) { return size_t(4 + 2 * D); }

// Test hooks of a decode call (null in every product call): the pipeline wait limit, and
// whether the copy of each split's first tile is withheld, so that the wait for it can only
// run out (nothing is in flight for it) and the bounded-wait failure path runs.
struct DecodeHooks {
  uint64_t wait_limit_ns;
  bool withhold_first_tile;
};

int plan_query_blocks(const rq_shape& s, int loop_begin, int loop_count, QueryBlock* out,
                      int max_out);

// Split kernel launches of a decode call.  When every block of the call is single-column
// (decode_combines_in_kernel), the last split of each (sequence, kv-head) combines into `out`
// (tickets: the call's cleared ticket region); otherwise tickets is null and the combine
// kernel follows.
bool decode_combines_in_kernel(const rq_shape& s, int loop_begin, int loop_count);
cudaError_t launch_rq_decode_mma(const rq_shape& s, const rq_cache& cache, const rq_paging* paging,
                                 const uint16_t* q, int loop_begin, int loop_count,
                                 const int32_t* ctx_lens, int n_splits, int tokens_per_split,
                                 const uint16_t* pending, uint16_t* out, float* part,
                                 unsigned* tickets, unsigned* err, cudaStream_t stream,
                                 const DecodeHooks* hooks = nullptr);

struct SplitPlan {
  int n_splits;          // split-KV partitions of the context
  int tokens_per_split;  // multiple of the kernel's token chunk
};

// Split-KV plan for a kernel that keeps `ctas_per_sm` CTAs resident per SM and moves
// `chunk`-token tiles: the number of splits minimises (waves) x (tiles per split + set-up).
SplitPlan plan_splits_for(const rq_shape& s, int max_ctx, int ctas_per_sm, int chunk);
SplitPlan plan_splits_rq(const rq_shape& s, int loop_begin, int loop_count, int max_ctx);
SplitPlan plan_splits_bf16(const rq_shape& s, int max_ctx);
SplitPlan plan_splits(const rq_shape& s, int loop_count, int max_ctx);
size_t partial_floats(const rq_shape& s);  // floats of one partial record

cudaError_t launch_encode(const rq_shape& s, const rq_cache& cache, const rq_paging* paging,
                          const uint16_t* kv_new,
                          const int64_t strides[5], const int32_t* positions, int32_t pos_begin,
                          int32_t n_new, cudaStream_t stream, int alpha_mode = 0);

cudaError_t launch_rq_decode(const rq_shape& s, const rq_cache& cache, const rq_paging* paging,
                             const uint16_t* q,
                             int loop_begin, int loop_count, const uint16_t* pending,
                             const int32_t* ctx_lens, int max_ctx, uint16_t* out, float* ws,
                             cudaStream_t stream, const DecodeHooks* hooks = nullptr);

cudaError_t launch_bf16_decode(const rq_shape& s, const uint16_t* k, const uint16_t* v,
                               const uint16_t* q, int loop_begin, int loop_count,
                               const uint16_t* pending, const int32_t* ctx_lens, int max_ctx,
                               uint16_t* out, float* ws, cudaStream_t stream);

cudaError_t launch_combine(const rq_shape& s, const int8_t* v_signs, const uint16_t* q,
                           int loop_count, const uint16_t* pending, int n_splits,
                           uint16_t* out, const float* part, const unsigned* err,
                           cudaStream_t stream);

// Ablation rows (include/rq_ablation.h): a per-loop decode call over a cache encoded with a
// fixed at 1 (mode 1) or 0 (mode 2), one query column per kv-head, head dim 128.
cudaError_t launch_rq_ablation_decode(const rq_shape& s, const rq_cache& cache, int mode,
                                      const uint16_t* q, int loop, const uint16_t* pending,
                                      const int32_t* ctx_lens, int max_ctx, uint16_t* out,
                                      float* ws, cudaStream_t stream);

int device_sm_count();

// The argument checks of rq_decode_attention other than its workspace (C ABI layer).
rq_status validate_decode(const rq_shape* shape, const rq_cache* cache, const uint16_t* q,
                          int32_t loop_begin, int32_t loop_count, const int32_t* ctx_lens,
                          int32_t max_ctx, uint16_t* out);

}  // namespace rq
