// ResidualQuant split-KV decode attention on the tensor cores (sm_103a): host side (query
// blocks, split plan, launches) and the contiguous-cache kernel variants.  The kernel itself
// is in rq_decode_mma.cuh.
#include <mutex>

#include "rq_decode_mma.cuh"

namespace rq {
namespace {


KernelFn pick(int D, bool res4, int nr, bool paged, int pk) {
  if (paged) return pick_paged(D, res4, nr, pk);
  if (pk == 2) return pick_pg<false, 2>(D, res4, nr);
  return pk == 1 ? pick_pg<false, 1>(D, res4, nr) : pick_pg<false, 0>(D, res4, nr);
}

// Opt every kernel variant in to the largest dynamic shared memory, once per device.
cudaError_t prepare_kernels() {
  static std::once_flag once[64];
  static cudaError_t err[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    err[dev] = cudaSuccess;
    for (int D : {64, 128})
      for (bool r4 : {false, true})
        for (int v = 0; v < 6; ++v)   // contiguous / paged, each with the three packings
          for (int nr = -1; nr <= kMaxResPerBlock; ++nr) {
            cudaError_t e = cudaFuncSetAttribute(pick(D, r4, nr, v >= 3, v % 3),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 200 * 1024);
            if (e != cudaSuccess) err[dev] = e;
          }
  });
  return err[dev];
}

// Packing of the MMA columns for a block: one query column -> its channel groups take the
// columns (2); at most 4 -> low parts in columns 4-7 (1); else high and low parts in two MMAs.
int block_packing(const QueryBlock& bq) {
  const int cols = bq.gw * bq.nl;
  return cols == 1 ? 2 : (cols <= 4 ? 1 : 0);
}

// CTAs of a kernel variant resident per SM with `smem` bytes of dynamic shared memory.
int resident_ctas(int D, bool res4, int nr, int pk, size_t smem) {
  int n = 0;
  if (prepare_kernels() == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pick(D, res4, nr, false, pk), kW * 32, smem) ==
          cudaSuccess &&
      n > 0)
    return n;
  const int by_smem = int((227 * 1024) / (smem + 1024));   // no device: shared-memory bound
  return by_smem < 1 ? 1 : (by_smem > 8 ? 8 : by_smem);
}

struct BlockLaunch {
  MmaArgs a;
  bool res4;
  size_t smem;
};

// Arguments, stage layout and shared memory of one query block (no launch).
bool build_block(const rq_shape& s, const rq_cache& cache, const QueryBlock& bq, int n_pg,
                 BlockLaunch& bl) {
  MmaArgs& a = bl.a;
  memset(&a, 0, sizeof(a));
  const int D = s.head_dim, NG = D / 32;
  a.data = cache.data;
  a.rec_bytes = record_bytes(s);
  // stage layout: the record's reference section, then the sections of the block's residual
  // loops (consecutive loops, consecutive sections), the same offsets as in the record
  int off = 0;
  a.off_kc = off; off += kT * D / 2;
  a.off_km = off; off += kT * NG * 4;
  a.off_vc = off; off += kT * D / 2;
  a.off_vm = off; off += kT * NG * 4;
  bool res4 = false;
  for (int ri = 0; ri < bq.nr; ++ri) {
    const int l = bq.r0 + ri;
    const int bits = s.res_bits[l];
    res4 |= bits == 4;
    a.rbits[ri] = bits;
    a.off_krc[ri] = off; off += kT * D * bits / 8;
    a.off_krm[ri] = off; off += kT * NG * 4;
    a.off_ka[ri] = off;  off += kT * 2;
    a.off_vrc[ri] = off; off += kT * D * bits / 8;
    a.off_vrm[ri] = off; off += kT * NG * 4;
    a.off_va[ri] = off;  off += kT * 2;
  }
  a.stage_bytes = off;
  const int refb = ref_section_bytes(D);
  a.cp_src[0] = 0;
  a.cp_dst[0] = 0;
  if (bq.nr == 0 || bq.r0 == 0) {   // the reference section (and loops 0 ..): one piece
    a.ncp = 1;
    a.cp_bytes[0] = off;
  } else {
    a.ncp = 2;
    a.cp_bytes[0] = refb;
    a.cp_src[1] = loop_section_offset(D, s.res_bits, bq.r0);
    a.cp_dst[1] = refb;
    a.cp_bytes[1] = off - refb;
  }
  a.qrm_bytes = masked_fragment_bytes(D, res4, bq.nr, block_packing(bq));
  a.blk = bq;
  a.n_pg = n_pg;
  bl.res4 = res4;
  // most resident CTAs per SM first (latency hiding), then the deepest pipeline
  int best_ctas = 0;
  for (int stages = 3; stages >= 2; --stages) {
    const size_t sm = smem_layout(D, res4, stages, a.stage_bytes, n_pg, a.qrm_bytes).total;
    if (sm > 200 * 1024) continue;
    const int ctas = resident_ctas(D, res4, bq.nr, block_packing(bq), sm);
    if (ctas > best_ctas) {
      best_ctas = ctas;
      a.n_stages = stages;
      bl.smem = sm;
    }
  }
  return best_ctas > 0;
}

}  // namespace

// Query columns per launch: one 8-column n-tile keeps registers and shared memory low enough
// for three resident CTAs per SM; wider blocks (which read the reference tile once for more
// loops) measured slower on GB300 because of the lower occupancy.
constexpr int kMaxBlockColumns = kNQ;

int plan_query_blocks(const rq_shape& s, int loop_begin, int loop_count, QueryBlock* out,
                      int max_out) {
  const int g = s.n_q_heads / s.n_kv_heads, L = s.n_loops;
  int gw = 1;
  while (gw < g && gw < 8) gw <<= 1;
  // One query head per kv-head and head dim 128: a 4-bit residual loop takes a single-column
  // block of its own, the other loops of the call share blocks.  (The multi-column variants
  // with a 4-bit loop hold more registers than three CTAs per SM allow without spilling; the
  // second read of the reference tile costs less.)
  const bool four_alone = gw == 1 && s.head_dim == 128;
  int n = 0;
  for (int gi0 = 0; gi0 < g; gi0 += gw) {
    int l = loop_begin;
    const int lend = loop_begin + loop_count;
    while (l < lend) {
      QueryBlock bq;
      bq.gi0 = gi0;
      bq.gw = gw;
      bq.lb = l;
      int nl = 0, nres = 0;
      while (l + nl < lend && (nl + 1) * gw <= kMaxBlockColumns) {
        const bool res = (l + nl) != L - 1;
        const bool four = res && s.res_bits[l + nl] == 4;
        if (res && nres == kMaxResPerBlock) break;
        if (four_alone && four && nl > 0) break;     // ends the block before it
        nres += res;
        ++nl;
        if (four_alone && four) break;               // and stands alone
      }
      bq.nl = nl;
      bq.r0 = l;
      bq.nr = nres;
      if (n >= max_out) return -1;
      out[n++] = bq;
      l += nl;
    }
  }
  return n;
}

bool decode_combines_in_kernel(const rq_shape& s, int loop_begin, int loop_count) {
  QueryBlock blocks[64];
  const int nb = plan_query_blocks(s, loop_begin, loop_count, blocks, 64);
  if (nb < 1) return false;
  for (int i = 0; i < nb; ++i) {
    const int nr = blocks[i].nr;
    bool res4 = false;
    for (int ri = 0; ri < nr; ++ri) res4 |= s.res_bits[blocks[i].r0 + ri] == 4;
    if (block_packing(blocks[i]) != 2 || !has_single_column_variant(s.head_dim, res4, nr)) return false;
  }
  return true;
}

SplitPlan plan_splits_rq(const rq_shape& s, int loop_begin, int loop_count, int max_ctx) {
  // the resident CTAs per SM follow the largest shared-memory block of the call
  QueryBlock blocks[64];
  const int nb = plan_query_blocks(s, loop_begin, loop_count, blocks, 64);
  rq_cache dummy;
  memset(&dummy, 0, sizeof(dummy));
  int ctas = 0;
  for (int i = 0; i < nb; ++i) {
    BlockLaunch bl;
    if (!build_block(s, dummy, blocks[i], 0, bl)) continue;
    const int n = resident_ctas(s.head_dim, bl.res4, blocks[i].nr, block_packing(blocks[i]), bl.smem);
    if (ctas == 0 || n < ctas) ctas = n;
  }
  return plan_splits_for(s, max_ctx, ctas > 0 ? ctas : 1, kT);
}

cudaError_t launch_rq_decode_mma(const rq_shape& s, const rq_cache& cache, const rq_paging* paging,
                                 const uint16_t* q, int loop_begin, int loop_count,
                                 const int32_t* ctx_lens, int n_splits, int tokens_per_split,
                                 const uint16_t* pending, uint16_t* out, float* part,
                                 unsigned* tickets, unsigned* err, cudaStream_t stream,
                                 const DecodeHooks* hooks) {
  cudaError_t e = prepare_kernels();
  if (e != cudaSuccess) return e;
  QueryBlock blocks[64];
  const int g = s.n_q_heads / s.n_kv_heads;
  const int nb = plan_query_blocks(s, loop_begin, loop_count, blocks, 64);
  if (nb < 0) return cudaErrorInvalidConfiguration;
  const float scale = s.softmax_scale > 0.f ? s.softmax_scale : 1.0f / sqrtf(float(s.head_dim));
  for (int bi = 0; bi < nb; ++bi) {
    BlockLaunch bl;
    const int n_pg = paging ? tokens_per_split / kT : 0;
    if (!build_block(s, cache, blocks[bi], n_pg, bl)) return cudaErrorInvalidConfiguration;
    MmaArgs& a = bl.a;
    a.bt = paging ? paging->block_table : nullptr;
    a.max_pages = paging ? paging->max_pages : 0;
    a.n_pages = paging ? paging->n_pages : 0;
    a.ksigns = cache.rot_signs[0];
    a.q = q;
    a.ctx_lens = ctx_lens;
    a.part = part;
    a.err = err;
    a.pending = pending;
    a.out = out;
    a.vsigns = cache.rot_signs[1];
    a.tickets = tickets ? tickets + int64_t(bi) * s.batch * s.n_kv_heads : nullptr;   // block's
    a.B = s.batch;
    a.Hq = s.n_q_heads;
    a.H = s.n_kv_heads;
    a.L = s.n_loops;
    a.cap = s.capacity;
    a.g = g;
    a.loop_begin = loop_begin;
    a.loop_count = loop_count;
    a.n_splits = n_splits;
    a.tokens_per_split = tokens_per_split;
    a.scale_log2 = scale * kLog2e;
    a.wait_limit_ns = hooks ? hooks->wait_limit_ns : kWaitLimitNs;
    a.withhold_first_tile = hooks && hooks->withhold_first_tile ? 1 : 0;
    dim3 grid(n_splits, s.n_kv_heads, s.batch);
    pick(s.head_dim, bl.res4, blocks[bi].nr, paging != nullptr, block_packing(blocks[bi]))<<<grid, kW * 32, bl.smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---------------------------------------------------------------------------- ablation rows
// Per-loop calls with one query column per kv-head and head dim 128 over a cache encoded with
// a fixed at 1 (mode 1, no a stream read) or at 0 (mode 2: the loop's own rotated INT2/INT4
// codes, no reference read): the single-column kernel with the reference and/or the a stream
// left out of its stage.

namespace {

template <int MODE>
KernelFn pick_mode(bool res4) {
  return res4 ? rq_mma_kernel<128, true, 1, false, 2, MODE> : rq_mma_kernel<128, false, 1, false, 2, MODE>;
}

}  // namespace

cudaError_t launch_rq_ablation_decode(const rq_shape& s, const rq_cache& cache, int mode,
                                      const uint16_t* q, int loop, const uint16_t* pending,
                                      const int32_t* ctx_lens, int max_ctx, uint16_t* out,
                                      float* ws, cudaStream_t stream) {
  const KernelFn fn = mode == 1 ? pick_mode<1>(s.res_bits[loop] == 4) : pick_mode<2>(s.res_bits[loop] == 4);
  const int D = 128, NG = 4;
  const int bits = s.res_bits[loop];
  MmaArgs a;
  memset(&a, 0, sizeof(a));
  a.data = cache.data;
  a.rec_bytes = record_bytes(s);
  const int refb = ref_section_bytes(D);
  const int rb = D * bits / 8;
  int off = 0;
  if (mode != 2) {   // the reference section (mode 1: the a rows come along, unread)
    a.off_kc = off; off += kT * D / 2;
    a.off_km = off; off += kT * NG * 4;
    a.off_vc = off; off += kT * D / 2;
    a.off_vm = off; off += kT * NG * 4;
  }
  a.rbits[0] = bits;
  a.off_krc[0] = off; off += kT * rb;
  a.off_krm[0] = off; off += kT * NG * 4;
  a.off_ka[0] = off;  off += kT * 2;
  a.off_vrc[0] = off; off += kT * rb;
  a.off_vrm[0] = off; off += kT * NG * 4;
  a.off_va[0] = off;  off += kT * 2;
  const int secoff = loop_section_offset(D, s.res_bits, loop);
  if (mode == 2) {            // the loop's section alone
    a.ncp = 1;
    a.cp_src[0] = secoff;
    a.cp_dst[0] = 0;
    a.cp_bytes[0] = off;
  } else if (loop == 0) {     // reference and loop 0: one piece
    a.ncp = 1;
    a.cp_bytes[0] = off;
  } else {
    a.ncp = 2;
    a.cp_bytes[0] = refb;
    a.cp_src[1] = secoff;
    a.cp_dst[1] = refb;
    a.cp_bytes[1] = off - refb;
  }
  a.stage_bytes = off;
  a.qrm_bytes = 0;
  QueryBlock bq;
  bq.gi0 = 0; bq.gw = 1; bq.lb = loop; bq.nl = 1; bq.r0 = loop; bq.nr = 1;
  a.blk = bq;
  // the method's split plan for this per-loop call (the workspace is sized for it)
  const SplitPlan plan = plan_splits_rq(s, loop, 1, max_ctx);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (e != cudaSuccess) return e;
  size_t smem = 0;
  int best = 0;
  for (int stages = 3; stages >= 2; --stages) {
    const size_t sm = smem_layout(D, bits == 4, stages, a.stage_bytes, 0, 0).total;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kW * 32, sm) != cudaSuccess) n = 0;
    if (n > best) {
      best = n;
      a.n_stages = stages;
      smem = sm;
    }
  }
  if (best == 0) return cudaErrorInvalidConfiguration;
  unsigned* err = reinterpret_cast<unsigned*>(ws);
  const size_t tb = ws_ticket_bytes(s, 1);
  unsigned* tickets = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(ws) + kWsHeaderBytes);
  float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + kWsHeaderBytes + tb);
  e = cudaMemsetAsync(ws, 0, kWsHeaderBytes + tb, stream);
  if (e != cudaSuccess) return e;
  a.ksigns = cache.rot_signs[0];
  a.vsigns = cache.rot_signs[1];
  a.q = q;
  a.ctx_lens = ctx_lens;
  a.part = part;
  a.err = err;
  a.pending = pending;
  a.out = out;
  a.tickets = tickets;
  a.B = s.batch;
  a.Hq = s.n_q_heads;
  a.H = s.n_kv_heads;
  a.L = s.n_loops;
  a.cap = s.capacity;
  a.g = 1;
  a.loop_begin = loop;
  a.loop_count = 1;
  a.n_splits = plan.n_splits;
  a.tokens_per_split = plan.tokens_per_split;
  const float scale = s.softmax_scale > 0.f ? s.softmax_scale : 1.0f / sqrtf(float(s.head_dim));
  a.scale_log2 = scale * kLog2e;
  a.wait_limit_ns = kWaitLimitNs;
  dim3 grid(plan.n_splits, s.n_kv_heads, s.batch);
  fn<<<grid, kW * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace rq
