// ResidualQuant split-KV decode attention on the tensor cores (sm_103a): the kernel
// template and its argument block, included by the translation units that instantiate it
// (rq_decode_mma.cu: contiguous cache, rq_decode_mma_paged.cu: paged cache).
//
// Per CTA: one (split of the context, kv-head, sequence) and one block of at most 8 query
// columns; 4 warps; 64-token tiles of every packed array are staged in shared memory by 1-D
// bulk (TMA) copies through a multi-stage mbarrier pipeline.  For a loop-l query q and token
// t (rit.work summary, "How each pass's KV cache is reconstructed": reference and residuals
// rebuilt inside attention)
//   score_t = a_t * sum_g [s^r_g,t (q_g . c^r_g,t) + z^r_g,t sum(q_g)]
//           +       sum_g [s^e_g,t (q'_g . c^e_g,t) + z^e_g,t sum(q'_g)],      q' = R q
//   acc_ref += p_t a_t (s^r c^r + z^r),   acc_res += p_t (s^e c^e + z^e)   (rotated domain)
//
// Each warp owns 16 tokens of every tile from scores to values, with its own online-softmax
// state, so no warp waits for another inside the loop:
//   scores: mma.sync m16n8k16, M = the warp's 16 tokens, N = 8 query columns, K = 16
//           channels; A = packed K codes, B = query fragments;
//   softmax: warp-local running max per column (raised lazily, only when a tile's maximum
//           exceeds it by more than 2^4 in probability), exponentials in the score fragment;
//   values: M = 16 channels, N = 8 columns, K = the warp's 16 tokens; A = packed V codes,
//           B = softmax weights p * a * step, moved from the score fragment's layout to the
//           B-operand layout in registers by movmatrix transposes.
// A stage is refilled by the last warp to finish with it; the four warps' partial results
// are merged once per CTA at the end.
//
// A pair of packed codes becomes an f16x2 operand with one AND (scores: the masked bits are
// the fp16 subnormal c * 2^-24 times a power of two fixed by their bit position, folded into
// the query fragments, with 2^24 restored in fp32) or with an OR and a packed subtraction
// (values: exact normal fp16 code times a power of two removed per output row at the end, for
// 4-bit codes; 2-bit residual codes are subnormal like the score operands, with 2^24 and the
// bit position's power of two removed per output row at the end).
// The other operand (queries, softmax weights) is split into an fp16 high part and an fp16
// low part (two MMAs; for blocks of at most 4 query columns one MMA, the low parts riding in
// the 4 free columns; for a single query column the columns carry its channel groups) and so
// carries about 22 significant bits; products are exact in the fp32 accumulators.
// Query columns of every loop share the fragments: the residual codes of loop l meet the
// query fragments of every column, and each column keeps only its own loop's dot product
// (a per-loop score accumulator, or a query fragment masked to the loop's columns); in the
// value phase the weights of loop l's residual codes are masked to loop l's columns.
#pragma once

#include "rq_common.cuh"
#include "rq_kernels.h"
#include "rq_ptx.cuh"

namespace rq {

constexpr int kT = 64;                        // tokens per tile
constexpr int kW = 4;                         // warps per CTA; warp w owns tokens [16w, 16w+16)
constexpr int kNQ = 8;                        // query columns of a block (one n-tile)
constexpr float kRescaleSlack = 4.f;          // log2 units: weights stay <= 2^4 between rescales
constexpr int kIssuedSlot = 15;               // release-counter word holding the tiles issued
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct MmaArgs {
  const uint8_t* data;       // tile records of the packed cache
  int64_t rec_bytes;         // bytes of one record
  int ncp;                   // pieces of a record a stage takes (1 or 2): source offset in
  int cp_src[2], cp_dst[2], cp_bytes[2];   // the record, offset in the stage, bytes
  int rbits[kMaxResPerBlock];
  const int8_t* ksigns;
  const uint16_t* q;
  const int32_t* ctx_lens;
  float* part;
  unsigned* err;
  const uint16_t* pending;   // current token's K/V rows, or null
  uint16_t* out;
  const int8_t* vsigns;      // V rotation signs [H][D]
  unsigned* tickets;         // [B][H] of this launch's block: splits stored (or null: the
                             // combine kernel merges the splits)
  int B, Hq, H, L, cap, g, loop_begin, loop_count, n_splits, tokens_per_split;
  QueryBlock blk;
  float scale_log2;
  int n_stages, stage_bytes;
  int qrm_bytes;             // masked rotated-query fragments (masked_fragment_bytes)
  uint64_t wait_limit_ns;     // pipeline wait limit (kWaitLimitNs in product calls)
  int withhold_first_tile;    // test hook: tile 0 of every split is never copied
  const int32_t* bt;   // block table of a paged cache, or null
  int max_pages, n_pages, n_pg;   // table columns, physical pages, page-id slots in shared memory
  int off_kc, off_km, off_vc, off_vm;
  int off_krc[kMaxResPerBlock], off_krm[kMaxResPerBlock], off_ka[kMaxResPerBlock];
  int off_vrc[kMaxResPerBlock], off_vrm[kMaxResPerBlock], off_va[kMaxResPerBlock];
};

using KernelFn = void (*)(MmaArgs);

namespace {

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

template <int N>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&w)[N]) {
  if constexpr (N == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x;
    w[1] = v.y;
  }
}

__device__ __forceinline__ float2 ld_meta(const uint8_t* p) {  // (step, offset) fp16 pair
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}

__device__ __forceinline__ float2 meta_f2(uint32_t w) {  // packed (step, offset) -> fp32
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

__device__ __forceinline__ float ld_half(const uint8_t* p) {
  return __half2float(*reinterpret_cast<const __half*>(p));
}

// arr[i] for a runtime i < kMaxResPerBlock without indexing the parameter array at run time
__device__ __forceinline__ int pick_int(const int (&arr)[kMaxResPerBlock], int i) {
  int v = arr[0];
#pragma unroll
  for (int k = 1; k < kMaxResPerBlock; ++k) v = (i == k) ? arr[k] : v;
  return v;
}

// m ? x : y for a mask m of all ones or all zeros, as bit operations (one LOP3)
__device__ __forceinline__ float blend(uint32_t m, float x, float y) {
  return __uint_as_float((__float_as_uint(x) & m) | (__float_as_uint(y) & ~m));
}

__device__ __forceinline__ uint4 sel4(bool keep, uint4 v) {
  return keep ? v : make_uint4(0u, 0u, 0u, 0u);
}

// Transpose of an 8x8 matrix of 16-bit values held one row-pair per lane (lane 4i + j holds
// row i, columns 2j and 2j+1): afterwards the lane holds row i, columns 2j, 2j+1 of the
// transpose.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_u32(p)), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 4-bit group row (16 bytes) of one token: the A-operand pairs of k-step s for this lane's
// word; slot order (2c, 2c+1 | 2c+8, 2c+9) <- channels (8c+2s, 8c+2s+4 | 8c+2s+1, 8c+2s+5),
// the second pair scaled by 16.
template <bool NORMAL = false>
__device__ __forceinline__ void a_pairs_4bit(uint32_t w, int s, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = s ? (w >> 8) : w;
  lo = NORMAL ? code_pair_normal(x, 0x000F000Fu) : code_pair(x, 0x000F000Fu);
  hi = NORMAL ? code_pair_normal(x, 0x00F000F0u) : code_pair(x, 0x00F000F0u);
}

// 2-bit group row (8 bytes): this lane's byte-half of word c/2; k-step s uses codes 2s and
// 2s+1 of each half (channels 16(c/2) + 4(c%2) + 2s + {0, 1} and +8), scaled by 4^(2s) and
// 4^(2s+1).
template <bool NORMAL = false>
__device__ __forceinline__ void a_pairs_2bit(uint32_t x, int s, uint32_t& lo, uint32_t& hi) {
  const uint32_t m0 = 0x00030003u << (4 * s), m1 = 0x00030003u << (4 * s + 2);
  lo = NORMAL ? code_pair_normal(x, m0) : code_pair(x, m0);
  hi = NORMAL ? code_pair_normal(x, m1) : code_pair(x, m1);
}

// Softmax weights of one channel group in the score-fragment layout (token rows tr0 = r and
// tr1 = r + 8 of the warp, columns 2c and 2c + 1) -> the B-operand pairs of the value MMA
// (tokens 2c, 2c+1 | 2c+8, 2c+9 of the warp, column r), split into fp16 high and low parts.
__device__ __forceinline__ void weights_to_b(float w00, float w01, float w10, float w11,
                                             uint32_t& bh0, uint32_t& bh1, uint32_t& bl0,
                                             uint32_t& bl1) {
  uint32_t hT, lT, hB, lB;
  split_half2(w00, w01, hT, lT);
  split_half2(w10, w11, hB, lB);
  bh0 = movmatrix_trans(hT);
  bh1 = movmatrix_trans(hB);
  bl0 = movmatrix_trans(lT);
  bl1 = movmatrix_trans(lB);
}

// Blocks with at most 4 query columns carry the low parts of the split in the MMA's columns
// 4-7: lanes holding columns 0-3 (fragment lanes c < 2) pass the high parts of their weights,
// lanes holding columns 4-7 the low parts of columns 0-3; one transpose per token half.
__device__ __forceinline__ void weights_to_b_packed(float w00, float w01, float w10, float w11,
                                                    bool low, uint32_t& b0, uint32_t& b1) {
  uint32_t hT, lT, hB, lB;
  split_half2(w00, w01, hT, lT);
  split_half2(w10, w11, hB, lB);
  b0 = movmatrix_trans(low ? lT : hT);
  b1 = movmatrix_trans(low ? lB : hB);
}

// NRT >= 0: the block's number of residual loops, fixed at compile time; -1: read at run time.
// PAGED: tiles are found through the block table of a paged cache.
// PK (packing of the MMA's 8 columns): 0 = up to 8 query columns, high and low parts of the
// splits in two MMAs; 1 = at most 4 query columns, the low parts of the query and weight splits
// ride in columns 4-7 (one MMA where two would be); 2 = one query column, whose channel groups
// take the columns: group g's high parts in column g, its low parts in column g + 4, so that
// every lane of a fragment row scales distinct groups and one transpose serves every group.
// Blocks of the final loop alone (NRT 0) and single-column blocks with a 2-bit residual loop
// are held to 128 registers for four resident CTAs per SM; the others take up to 168 for three.
// MODE (ablation rows of the method's steps; single-column blocks of one residual loop only):
// 0 = the method; 1 = a fixed at 1 (the a rows are not read); 2 = direct quantisation of the
// loop (the reference is neither copied nor read: the score and the value are the loop's own
// codes alone, a = 0).
template <int D, bool RES4, int NRT, bool PAGED, int PK, int MODE = 0>
__global__ void __launch_bounds__(kW * 32, (NRT == 0 || (PK == 2 && !RES4)) ? 4 : 3) rq_mma_kernel(const __grid_constant__ MmaArgs a) {
  constexpr int NG = D / 32;
  constexpr int NQ = kNQ;
  constexpr int P = D / 32;          // channels per lane in the query prep
  constexpr int RB4 = D / 2;         // bytes of a 4-bit row
  constexpr int RB2 = D / 4;         // bytes of a 2-bit row
  constexpr int MT = D / 16;         // 16-channel m-tiles of the value phase (2 per group)
  constexpr bool PER_LOOP = NRT >= 1 && NRT <= 3;   // one residual score accumulator per loop
  constexpr bool HL = PK >= 1;                      // low parts in columns 4-7
  constexpr bool SC = PK == 2;                      // one query column, groups in columns
  // 4-column packing with 2 or 3 residual loops of 2 bits: each loop's residual MMAs take the
  // rotated-query fragments masked to its columns (no per-loop accumulator to select from)
  constexpr bool MASKB = (PK == 1 || PK == 0) && !RES4 && PER_LOOP && NRT >= 2;
  static_assert(!SC || (NRT == 0 || NRT == 1) && D == 128, "single-column blocks: D 128, one loop");
  static_assert(MODE == 0 || (SC && NRT == 1 && !PAGED), "ablation modes: single-column, one loop");
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const QueryBlock blk = a.blk;
  const int nr = NRT >= 0 ? NRT : blk.nr;

  // Stage layout (byte offsets within a stage, the order of the cache's tile records): K
  // codes, K steps, V codes, V steps, then per residual loop K codes, K steps, K a, V codes,
  // V steps, V a.  Fixed at compile time when the residual-loop count is and every residual
  // loop is 2-bit (the run-time offsets cost registers and constant-bank loads in the loop;
  // 8-column blocks of three loops keep them: the constants spill there).
  constexpr bool FIXED = MODE != 2 && !RES4 && NRT >= 0 && (NRT <= 2 || (NRT == 3 && PK == 1));
  constexpr int F_KM = kT * RB4, F_VC = F_KM + kT * NG * 4, F_VM = F_VC + kT * RB4;
  constexpr int F_RES = F_VM + kT * NG * 4;
  constexpr int F_KRM = kT * RB2, F_KA = F_KRM + kT * NG * 4, F_VRC = F_KA + kT * 2;
  constexpr int F_VRM = F_VRC + kT * RB2, F_VA = F_VRM + kT * NG * 4, F_RS = F_VA + kT * 2;
  const int o_kc = FIXED ? 0 : a.off_kc;
  const int o_km = FIXED ? F_KM : a.off_km;
  const int o_vc = FIXED ? F_VC : a.off_vc;
  const int o_vm = FIXED ? F_VM : a.off_vm;
  const int SB = FIXED ? F_RES + (NRT >= 0 ? NRT : 0) * F_RS : a.stage_bytes;
  auto o_krc = [&](int ri) { return FIXED ? F_RES + ri * F_RS : a.off_krc[ri]; };
  auto o_vrc = [&](int ri) { return FIXED ? F_RES + ri * F_RS + F_VRC : a.off_vrc[ri]; };

  // Single-column blocks combine their splits in the kernel: the last split of this
  // (sequence, kv-head) to store its records merges every split's records, adds the current
  // token and undoes the rotation (the stores of the other splits are ordered before their
  // ticket by a fence, and the ticket before the reads).  Other blocks leave that to the
  // combine kernel: for them the fence at every CTA's end and the combine on the tail cost
  // more than the launch it saves.
  auto combine_if_last = [&]() {
    if constexpr (!SC) return;
    if (!a.tickets) return;   // (a call with other blocks: the combine kernel merges)
    __syncthreads();
    bool last = false;
    if (threadIdx.x == 0) {
      __threadfence();
      last = atomicAdd(&a.tickets[int64_t(b) * a.H + h], 1u) == unsigned(a.n_splits - 1);
    }
    if (!__syncthreads_or(last)) return;
    __threadfence();
    const bool gave_up = *reinterpret_cast<volatile const unsigned*>(a.err) != 0u;
    constexpr int rec = int(partial_floats_d(D));
    for (int col = warp; col < NQ; col += kW) {
      const int li = col / blk.gw, gi = blk.gi0 + col % blk.gw;
      if (li >= blk.nl || gi >= a.g) continue;
      const int lc = blk.lb + li - a.loop_begin;
      const int64_t wid = (int64_t(b) * a.Hq + int64_t(h) * a.g + gi) * a.loop_count + lc;
      const uint16_t* kpp = nullptr;
      const uint16_t* vpp = nullptr;
      if (a.pending) {
        kpp = a.pending + ((int64_t(b) * 2 + 0) * a.loop_count + lc) * a.H * D + int64_t(h) * D;
        vpp = a.pending + ((int64_t(b) * 2 + 1) * a.loop_count + lc) * a.H * D + int64_t(h) * D;
      }
      combine_column<D>(a.part + wid * a.n_splits * rec, a.n_splits, a.q + wid * D, kpp, vpp,
                        a.vsigns + int64_t(h) * D, a.scale_log2, gave_up, a.out + wid * D, lane);
    }
  };

  if (FIXED && SB != a.stage_bytes) {   // host and kernel disagree on the layout: refuse
    if (threadIdx.x == 0) atomicOr(a.err, 1u);
    combine_if_last();                  // (NaN outputs)
    return;
  }
  const int qrm_bytes = masked_fragment_bytes(D, RES4, NRT, PK);
  if (a.qrm_bytes != qrm_bytes || (qrm_bytes > 0) != MASKB) {   // layouts disagree: refuse
    if (threadIdx.x == 0) atomicOr(a.err, 1u);
    combine_if_last();
    return;
  }
  const SmemLayout lay = smem_layout(D, RES4, a.n_stages, SB, a.n_pg, qrm_bytes);
  uint4* QF = reinterpret_cast<uint4*>(smem + lay.qf);
  uint4* QR2 = reinterpret_cast<uint4*>(smem + lay.qr2);
  uint4* QR4 = reinterpret_cast<uint4*>(smem + lay.qr4);
  float* Qsum = reinterpret_cast<float*>(smem + lay.qsum);
  float* QRsum = reinterpret_cast<float*>(smem + lay.qrsum);
  float* red = reinterpret_cast<float*>(smem + lay.red);      // [2][kW][NQ]
  unsigned* cnt = reinterpret_cast<unsigned*>(smem + lay.cnt);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  int* pid = reinterpret_cast<int*>(smem + lay.pg);   // physical page of each tile (paged)

  // residual index (into the block's residual loops) of query column n, -1 if the column
  // is the final loop's or a padding column
  auto col_ri = [&](int n) -> int {
    const int li = n / blk.gw, gi = blk.gi0 + n % blk.gw;
    const int l = blk.lb + li;
    return (li < blk.nl && gi < a.g && l != a.L - 1) ? l - blk.r0 : -1;
  };

  // ------------------------------------------------------------------ pipeline set-up
  // (first: the first tiles stream in while the queries are prepared)
  const int ctx_raw = a.ctx_lens[b];
  const int ctx = min(ctx_raw, a.cap);
  const int t_begin = split * a.tokens_per_split;
  // a context longer than the call's splits cover (ctx_len above max_ctx or the capacity) or
  // negative is refused: the call is flagged (outputs NaN) rather than silently truncated
  if (split == a.n_splits - 1 && threadIdx.x == 0 &&
      (ctx_raw < 0 || ctx_raw > a.cap || int64_t(ctx_raw) > int64_t(a.n_splits) * a.tokens_per_split))
    atomicOr(a.err, 1u);
  const int t_end = min(ctx, t_begin + a.tokens_per_split);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kT - 1) / kT : 0;
  const int64_t slot = int64_t(b) * a.H + h;
  const int S = a.n_stages;
  constexpr bool paged = PAGED;
  // physical page of the split's tile (a paged cache's tiles are its 64-token pages); a
  // table entry out of range is never dereferenced: page 0 is read and the call flagged
  auto page_of = [&](int tile) -> int {
    int pg = a.bt[int64_t(b) * a.max_pages + t_begin / kT + tile];
    if (pg < 0 || pg >= a.n_pages) {
      atomicOr(a.err, 1u);
      pg = 0;
    }
    return pg;
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      cnt[s] = 0u;
    }
    fence_mbar_init();
  }

  // A stage is one or two contiguous pieces of the tile's record (the reference section and
  // the sections of the block's residual loops), one bulk copy each.
  auto issue = [&](int tile) {
    if (a.withhold_first_tile && tile == 0) return;   // (test hook: the wait can only run out)
    const int st = tile % S;
    const uint32_t bar = smem_u32(&bars[st]);
    const uint32_t dst = smem_u32(smem + st * a.stage_bytes);
    const int64_t rec = paged ? int64_t(pid[tile]) * a.H + h
                              : slot * (a.cap / kT) + t_begin / kT + tile;
    const uint8_t* src = a.data + rec * a.rec_bytes;
    mbar_arrive_expect_tx(bar, uint32_t(a.stage_bytes));
    bulk_g2s(dst + a.cp_dst[0], src + a.cp_src[0], uint32_t(a.cp_bytes[0]), bar);
    if (a.ncp > 1) bulk_g2s(dst + a.cp_dst[1], src + a.cp_src[1], uint32_t(a.cp_bytes[1]), bar);
  };
  if (threadIdx.x == 0) {   // the barriers' initialisation is ordered before by the fence
    const int n0 = S < ntiles ? S : ntiles;
    if (paged)
      for (int i = 0; i < n0; ++i) pid[i] = page_of(i);
    for (int i = 0; i < n0; ++i) issue(i);
    cnt[kIssuedSlot] = unsigned(n0);
  }

  // ------------------------------------------------------------------ query preparation
  // query columns of this block, two per warp: scaled q, rotated q' = R q, per-group sums
  auto prep_column = [&](int n, float (&v)[P], float (&rr)[P]) {
    const int li = n / blk.gw;
    const int gi = blk.gi0 + n % blk.gw;
    const bool real = li < blk.nl && gi < a.g;
    const int l = blk.lb + li;
    const int8_t* sg = a.ksigns + int64_t(h) * D + lane * P;
    if (real) {
      const uint16_t* qp =
          a.q + ((int64_t(b) * a.Hq + int64_t(h) * a.g + gi) * a.loop_count + (l - a.loop_begin)) * D +
          lane * P;
#pragma unroll
      for (int j = 0; j < P; ++j) v[j] = bf16_bits_to_float(qp[j]) * a.scale_log2;
    } else {
#pragma unroll
      for (int j = 0; j < P; ++j) v[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < P; ++j) rr[j] = v[j] * float(sg[j]);
    warp_fwht<P>(rr, lane);
    const float inv_sqrt_d = (D == 128) ? 0.08838834764831845f : 0.125f;
#pragma unroll
    for (int j = 0; j < P; ++j) rr[j] *= inv_sqrt_d;
  };
  constexpr int NCW = NQ / kW;                 // query columns per warp
  float qv[NCW][P], qr[NCW][P];
#pragma unroll
  for (int k = 0; k < NCW; ++k) prep_column(warp + k * kW, qv[k], qr[k]);
  {
    uint32_t* z32 = reinterpret_cast<uint32_t*>(smem + lay.qf);
    const int nz = (lay.cnt - lay.qf) / 4;
    for (int i = threadIdx.x; i < nz; i += blockDim.x) z32[i] = 0u;
    if (paged)   // the pages of the later tiles, read before the first refill needs them
      for (int i = S + threadIdx.x; i < ntiles; i += blockDim.x) pid[i] = page_of(i);
  }
  __syncthreads();
  // the largest |q|, |q'| of the block fixes a power-of-two fragment scale 2^k with
  // max |fragment| <= 2^14, so the low parts of the split stay normal fp16 (they meet the
  // subnormal code operands of the score MMAs)
  {
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < NCW; ++k)
#pragma unroll
      for (int j = 0; j < P; ++j) mx = fmaxf(mx, fmaxf(fabsf(qv[k][j]), fabsf(qr[k][j])));
    mx = warp_max(mx);
    if (lane == 0) atomicMax(reinterpret_cast<unsigned*>(red), __float_as_uint(mx));
  }
  __syncthreads();
  const float qmax = __uint_as_float(*reinterpret_cast<const unsigned*>(red));
  int qexp = 0;
  if (qmax > 0.f) {
    frexpf(qmax, &qexp);                     // qmax < 2^qexp
    qexp = 14 - qexp;
    qexp = qexp < 0 ? 0 : (qexp > 40 ? 40 : qexp);
  }
  const float qscale = ldexpf(1.f, qexp);
  const float code_unit = ldexpf(1.f, 24 - qexp);   // undoes 2^-24 codes and the q scale
  const float inv_code_unit = ldexpf(1.f, qexp - 24);
  // fragments and group sums (the sums in units of code_unit, which scales the score once at
  // the end)
#pragma unroll
  for (int k = 0; k < NCW; ++k) {
    const int n = warp + k * kW;
    const float (&v)[P] = qv[k];
    const float (&rr)[P] = qr[k];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      s1 += v[j];
      s2 += rr[j];
    }
#pragma unroll
    for (int o = 1; o < 32 / P; o <<= 1) {
      s1 += __shfl_xor_sync(RQ_FULL_MASK, s1, o);
      s2 += __shfl_xor_sync(RQ_FULL_MASK, s2, o);
    }
    const int ri = col_ri(n);
    const int bits = ri >= 0 ? a.rbits[ri] : 0;
    const int grp = (lane * P) >> 5;
    if ((lane & (32 / P - 1)) == 0 && !(HL && n >= 4)) {
      Qsum[grp * NQ + n] = s1 * inv_code_unit;
      if (ri >= 0) QRsum[grp * NQ + n] = s2 * inv_code_unit;
    }
    // (HL: the low part goes to column n + 4's entry, and columns 4-7 write nothing)
#pragma unroll
    for (int j = 0; j < P; ++j) {
      if (HL && n >= 4) break;
      if (SC && n != 0) break;       // (SC: columns 1-7 are the groups' slots)
      const int ch = lane * P + j, gq = ch >> 5, cl = ch & 31;
      const int ns = SC ? gq : n;    // fragment column of the high part
      const float vq = v[j] * qscale, rq = rr[j] * qscale;
      {  // 4-bit mapping: slot (c4, s, hi, e) <- channel 8 c4 + 2 s + hi + 4 e, scale 16^-hi
        const int c4 = cl >> 3, w8 = cl & 7, s = (w8 >> 1) & 1, hi = w8 & 1, e = w8 >> 2;
        const int idx = (gq * 2 + s) * 32 + ns * 4 + c4;
        __half* dq = reinterpret_cast<__half*>(&QF[idx]);
        __half* dql = HL ? reinterpret_cast<__half*>(&QF[idx + 16]) : dq + 4;
        split_half(hi ? vq * 0.0625f : vq, dq[hi * 2 + e], dql[hi * 2 + e]);
        if (RES4 && bits == 4) {
          __half* dr = reinterpret_cast<__half*>(&QR4[idx]);
          __half* drl = HL ? reinterpret_cast<__half*>(&QR4[idx + 16]) : dr + 4;
          split_half(hi ? rq * 0.0625f : rq, dr[hi * 2 + e], drl[hi * 2 + e]);
        }
      }
      if (bits == 2) {  // 2-bit mapping: slot (cq, s, hi, e) <- channel 16(cq/2)+4(cq%2)+2s+hi+8e
        const int e = (cl >> 3) & 1, cq = 2 * (cl >> 4) + ((cl & 7) >> 2), jj = cl & 3;
        const int s = jj >> 1, hi = jj & 1;
        const float sc = (jj == 0) ? 1.f : (jj == 1) ? 0.25f : (jj == 2) ? 0.0625f : 0.015625f;
        const int idx = (gq * 2 + s) * 32 + ns * 4 + cq;
        __half* dr = reinterpret_cast<__half*>(&QR2[idx]);
        __half* drl = HL ? reinterpret_cast<__half*>(&QR2[idx + 16]) : dr + 4;
        split_half(rq * sc, dr[hi * 2 + e], drl[hi * 2 + e]);
      }
    }
  }
  __syncthreads();   // fragments and sums visible to every warp

  // Offset terms of the scores, sum_g z_g,t sum(q_g), as one m16n8k8 MMA per reference or
  // residual loop and tile: A = the (step, offset) fp16 words of a token's 4 groups as stored,
  // B = 0 against the steps and the column's group sums against the offsets (scaled by 2^19,
  // which bounds them by 2^14 given the fragment scale, as fp16 high and low parts).  B slots:
  // 0/1 reference high/low, 2 + 2 ri / 3 + 2 ri residual loop ri (masked to its columns);
  // with the 4-column packing the low parts sit in columns 4-7 of the even slots.  Used for
  // blocks of at most one residual loop and for 4-column blocks; 8-column blocks with more
  // residual loops keep the per-element form (the added live registers cost spills there).
  constexpr bool OFS = !SC && NRT >= 0 && (NRT <= 1 || PK == 1);
  constexpr float kOfsScale = 524288.f, kOfsUnscale = 1.f / 524288.f;
  const uint32_t* OB = reinterpret_cast<const uint32_t*>(smem + lay.ob);
  if constexpr (OFS) {
    uint32_t* ob = reinterpret_cast<uint32_t*>(smem + lay.ob);
    for (int i = threadIdx.x; i < 8 * 32; i += kW * 32) {
      const int j = i >> 5, rr = (i & 31) >> 2, cc = i & 3;
      const int slot = j >> 1;             // 0: reference, 1 + ri: residual loop ri
      const bool low = HL ? rr >= 4 : (j & 1) != 0;
      const int col = HL ? (rr & 3) : rr;
      float v = 0.f;
      if (cc < NG && !(HL && (j & 1)) &&
          (slot == 0 || (slot - 1 < (NRT > 3 ? 3 : NRT) && col_ri(col) == slot - 1)))
        v = (slot == 0 ? Qsum : QRsum)[cc * NQ + col] * kOfsScale;
      __half hi, lw;
      split_half(v, hi, lw);
      ob[i] = uint32_t(__half_as_ushort(low ? lw : hi)) << 16;
    }
    __syncthreads();
  }
  const int cw = c < NG ? c : 0;   // this lane's group in the offset MMAs' A operand
  // masked fragments: [ri][k-step][lane], the rotated-query fragment where the lane's column
  // (4-column packing: high or low part of query column (lane / 4) & 3; 8 columns: query
  // column lane / 4, high and low parts) is residual loop ri's, else zero
  uint2* QRM = reinterpret_cast<uint2*>(smem + lay.qrm);
  uint4* QRM4 = reinterpret_cast<uint4*>(smem + lay.qrm);
  if constexpr (MASKB) {
    for (int i = threadIdx.x; i < NRT * NG * 2 * 32; i += kW * 32) {
      const int ri = i / (NG * 2 * 32), rem = i % (NG * 2 * 32);
      if constexpr (HL) {
        const uint2 v = *reinterpret_cast<const uint2*>(&QR2[rem]);
        QRM[i] = col_ri(((rem & 31) >> 2) & 3) == ri ? v : make_uint2(0u, 0u);
      } else {
        QRM4[i] = col_ri((rem & 31) >> 2) == ri ? QR2[rem] : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    __syncthreads();
  }

  // columns of this lane: score/value-accumulator fragments hold columns 2c and 2c + 1, the
  // value B operand column r
  int riD[2], krmD[2], kaD[2], vaD[2], vrmD[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    riD[e] = col_ri(HL ? (2 * c + e) & 3 : 2 * c + e);   // HL: the column whose low parts these are
    // (one residual loop: both columns' metadata is the same loop's, at a constant address,
    // so it is loaded and converted once)
    const int rc = (NRT == 1 || riD[e] < 0) ? 0 : riD[e];
    krmD[e] = FIXED ? F_RES + rc * F_RS + F_KRM : pick_int(a.off_krm, rc);
    kaD[e] = FIXED ? F_RES + rc * F_RS + F_KA : pick_int(a.off_ka, rc);
    vaD[e] = FIXED ? F_RES + rc * F_RS + F_VA : pick_int(a.off_va, rc);
    vrmD[e] = FIXED ? F_RES + rc * F_RS + F_VRM : pick_int(a.off_vrm, rc);
  }
  const int riB = col_ri(HL ? r & 3 : r);
  const bool low_lane = HL && c >= 2;   // fragment columns 4-7: low parts
  // SC: fragment columns 2c + e hold group gp + e (lanes c >= 2 its low parts); the offset
  // terms of the scores take the group sums in the high lanes only
  const int gp = 2 * (c & 1);
  float qsS[2] = {0.f, 0.f}, qrsS[2] = {0.f, 0.f};
  if constexpr (SC) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (!low_lane) {
        qsS[e] = Qsum[(gp + e) * NQ];
        if (NRT == 1) qrsS[e] = QRsum[(gp + e) * NQ];
      }
  }
  // loop_mask[e][ri]: all ones where column 2c + e belongs to residual loop ri
  uint32_t loop_mask[2][PER_LOOP ? NRT : 1];
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int ri = 0; ri < (PER_LOOP ? NRT : 1); ++ri) loop_mask[e][ri] = riD[e] == ri ? ~0u : 0u;

  float accR[MT][4], accE2[MT][4], accE4[RES4 ? MT : 1][4];
  float offR[NG][2], offE[NG][2];
  float lsum[2] = {0.f, 0.f}, mw[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      accR[m][k] = 0.f;
      accE2[m][k] = 0.f;
      if (RES4) accE4[m][k] = 0.f;
    }
#pragma unroll
  for (int g = 0; g < NG; ++g) offR[g][0] = offR[g][1] = offE[g][0] = offE[g][1] = 0.f;

  bool failed = false;
  const int tr0 = 16 * warp + r, tr1 = tr0 + 8;       // this lane's token rows in a tile
  const int p0 = 8 * warp + c, p1 = p0 + 4;           // token pairs of its value B rows
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % S;
    if (!__all_sync(RQ_FULL_MASK,
                    mbar_wait_bounded(smem_u32(&bars[st]), uint32_t((i / S) & 1), a.wait_limit_ns))) {
      failed = true;
      break;
    }
    const uint8_t* sb = smem + st * SB;
    const int t0 = t_begin + i * kT;
    if (t0 + 16 * warp < t_end) {   // the warp has tokens in this tile
      const bool v0 = t0 + tr0 < t_end, v1 = t0 + tr1 < t_end;
      const bool partial = t0 + 16 * warp + 16 > t_end;   // the warp's rows run past the context

      // ---------------------------------------------------------------- scores
      float sc[4];
      if constexpr (SC) {
        // one accumulator for every group: column n holds group n & 3 (n >= 4: low parts)
        float D0[4] = {0.f, 0.f, 0.f, 0.f}, Dr[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (MODE != 2) {
          uint32_t kw0[NG], kw1[NG];
          load_words<NG>(sb + o_kc + tr0 * RB4 + c * NG * 4, kw0);
          load_words<NG>(sb + o_kc + tr1 * RB4 + c * NG * 4, kw1);
#pragma unroll
          for (int gq = 0; gq < NG; ++gq)
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              uint32_t a0, a2, a1, a3;
              a_pairs_4bit(kw0[gq], s, a0, a2);
              a_pairs_4bit(kw1[gq], s, a1, a3);
              const uint2 bq = *reinterpret_cast<const uint2*>(&QF[(gq * 2 + s) * 32 + lane]);
              mma_f16(D0, a0, a1, a2, a3, bq.x, bq.y);
            }
        }
        if (NRT == 1) {   // the block's residual loop
          const bool two = !RES4 || a.rbits[0] == 2;
#pragma unroll
          for (int gq = 0; gq < NG; ++gq) {
            uint32_t wl, wh;
            if (two) {
              const int off = o_krc(0) + ((c >> 1) * NG + gq) * 4;
              wl = lds32(sb + off + tr0 * RB2) >> (8 * (c & 1));
              wh = lds32(sb + off + tr1 * RB2) >> (8 * (c & 1));
            } else {
              const int off = o_krc(0) + (c * NG + gq) * 4;
              wl = lds32(sb + off + tr0 * RB4);
              wh = lds32(sb + off + tr1 * RB4);
            }
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              uint32_t a0, a1, a2, a3;
              if (two) {
                a_pairs_2bit(wl, s, a0, a2);
                a_pairs_2bit(wh, s, a1, a3);
              } else {
                a_pairs_4bit(wl, s, a0, a2);
                a_pairs_4bit(wh, s, a1, a3);
              }
              const int fi = (gq * 2 + s) * 32 + lane;
              const uint2 bq = *reinterpret_cast<const uint2*>((RES4 && !two) ? &QR4[fi] : &QR2[fi]);
              mma_f16(Dr, a0, a1, a2, a3, bq.x, bq.y);
            }
          }
        }
        // step and offset of this lane's two groups for tokens tr0 and tr1
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (MODE != 2) {
          const uint2 m0 = *reinterpret_cast<const uint2*>(sb + o_km + (tr0 * NG + gp) * 4);
          const uint2 m1 = *reinterpret_cast<const uint2*>(sb + o_km + (tr1 * NG + gp) * 4);
          const float2 s00 = meta_f2(m0.x), s01 = meta_f2(m0.y);
          const float2 s10 = meta_f2(m1.x), s11 = meta_f2(m1.y);
          x[0] = fmaf(s00.x, D0[0], s00.y * qsS[0]);
          x[1] = fmaf(s01.x, D0[1], s01.y * qsS[1]);
          x[2] = fmaf(s10.x, D0[2], s10.y * qsS[0]);
          x[3] = fmaf(s11.x, D0[3], s11.y * qsS[1]);
        }
        if (NRT == 1) {   // a_t * reference part + residual part
          const uint2 r0 = *reinterpret_cast<const uint2*>(sb + krmD[0] + (tr0 * NG + gp) * 4);
          const uint2 r1 = *reinterpret_cast<const uint2*>(sb + krmD[0] + (tr1 * NG + gp) * 4);
          float al0 = 1.f, al1 = 1.f;   // (MODE 1: a = 1; MODE 2: no reference part)
          if constexpr (MODE == 0) {
            al0 = ld_half(sb + kaD[0] + tr0 * 2);
            al1 = ld_half(sb + kaD[0] + tr1 * 2);
          }
          const float2 t00 = meta_f2(r0.x), t01 = meta_f2(r0.y);
          const float2 t10 = meta_f2(r1.x), t11 = meta_f2(r1.y);
          x[0] = fmaf(al0, x[0], fmaf(t00.x, Dr[0], t00.y * qrsS[0]));
          x[1] = fmaf(al0, x[1], fmaf(t01.x, Dr[1], t01.y * qrsS[1]));
          x[2] = fmaf(al1, x[2], fmaf(t10.x, Dr[2], t10.y * qrsS[0]));
          x[3] = fmaf(al1, x[3], fmaf(t11.x, Dr[3], t11.y * qrsS[1]));
        }
        // the token's score: its groups and parts over the 4 lanes of the row
        float s_0 = x[0] + x[1], s_1 = x[2] + x[3];
        s_0 += __shfl_xor_sync(RQ_FULL_MASK, s_0, 1);
        s_1 += __shfl_xor_sync(RQ_FULL_MASK, s_1, 1);
        s_0 += __shfl_xor_sync(RQ_FULL_MASK, s_0, 2);
        s_1 += __shfl_xor_sync(RQ_FULL_MASK, s_1, 2);
        sc[0] = sc[1] = v0 ? s_0 * code_unit : -INFINITY;
        sc[2] = sc[3] = v1 ? s_1 * code_unit : -INFINITY;
      } else {
        float R[4], E[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) R[k] = E[k] = 0.f;
        if constexpr (OFS) {   // the offset terms: one MMA per loop (two without packing)
          uint32_t w0 = lds32(sb + o_km + (tr0 * NG + cw) * 4);
          uint32_t w1 = lds32(sb + o_km + (tr1 * NG + cw) * 4);
          if (NG < 4 && c >= NG) w0 = w1 = 0u;
          mma_f16_k8(R, w0, w1, OB[lane]);
          if (!HL) mma_f16_k8(R, w0, w1, OB[32 + lane]);
          if constexpr (PER_LOOP) {
#pragma unroll
            for (int ri = 0; ri < (PER_LOOP ? NRT : 1); ++ri) {
              const int ob0 = FIXED ? F_RES + ri * F_RS + F_KRM : a.off_krm[ri];
              uint32_t v0w = lds32(sb + ob0 + (tr0 * NG + cw) * 4);
              uint32_t v1w = lds32(sb + ob0 + (tr1 * NG + cw) * 4);
              if (NG < 4 && c >= NG) v0w = v1w = 0u;
              mma_f16_k8(E, v0w, v1w, OB[(2 + 2 * ri) * 32 + lane]);
              if (!HL) mma_f16_k8(E, v0w, v1w, OB[(3 + 2 * ri) * 32 + lane]);
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            R[k] *= kOfsUnscale;
            E[k] *= kOfsUnscale;
          }
        }
        uint32_t km0[NG], km1[NG], kw0[NG], kw1[NG];
        load_words<NG>(sb + o_km + tr0 * NG * 4, km0);
        load_words<NG>(sb + o_km + tr1 * NG * 4, km1);
        // this lane's word of every group (K rows are group-interleaved: one load)
        load_words<NG>(sb + o_kc + tr0 * RB4 + c * NG * 4, kw0);
        load_words<NG>(sb + o_kc + tr1 * RB4 + c * NG * 4, kw1);
#pragma unroll
        for (int gq = 0; gq < NG; ++gq) {
          {  // reference
            float Dg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              uint32_t a0, a2, a1, a3;
              a_pairs_4bit(kw0[gq], s, a0, a2);
              a_pairs_4bit(kw1[gq], s, a1, a3);
              if constexpr (HL) {
                const uint2 bq = *reinterpret_cast<const uint2*>(&QF[(gq * 2 + s) * 32 + lane]);
                mma_f16(Dg, a0, a1, a2, a3, bq.x, bq.y);
              } else {
                const uint4 bq = QF[(gq * 2 + s) * 32 + lane];
                mma_f16(Dg, a0, a1, a2, a3, bq.x, bq.y);
                mma_f16(Dg, a0, a1, a2, a3, bq.z, bq.w);
              }
            }
            const float2 m0 = meta_f2(km0[gq]), m1 = meta_f2(km1[gq]);
            if constexpr (OFS) {   // offsets: above
              R[0] = fmaf(m0.x, Dg[0], R[0]);
              R[1] = fmaf(m0.x, Dg[1], R[1]);
              R[2] = fmaf(m1.x, Dg[2], R[2]);
              R[3] = fmaf(m1.x, Dg[3], R[3]);
            } else {
              const float2 qs = *reinterpret_cast<const float2*>(&Qsum[gq * NQ + 2 * c]);
              R[0] = fmaf(m0.x, Dg[0], fmaf(m0.y, qs.x, R[0]));
              R[1] = fmaf(m0.x, Dg[1], fmaf(m0.y, qs.y, R[1]));
              R[2] = fmaf(m1.x, Dg[2], fmaf(m1.y, qs.x, R[2]));
              R[3] = fmaf(m1.x, Dg[3], fmaf(m1.y, qs.y, R[3]));
            }
          }
          if (nr > 0) {  // residuals of every loop of the block
            float dsel[4];
            if constexpr (PER_LOOP) {
#pragma unroll
              for (int k = 0; k < 4; ++k) dsel[k] = 0.f;
#pragma unroll
              for (int ri = 0; ri < NRT; ++ri) {
                float Dr[4] = {0.f, 0.f, 0.f, 0.f};
                const bool two = !RES4 || a.rbits[ri] == 2;   // without 4-bit loops: all 2-bit
                uint32_t wl, wh;
                if (two) {
                  const int off = o_krc(ri) + ((c >> 1) * NG + gq) * 4;
                  wl = lds32(sb + off + tr0 * RB2) >> (8 * (c & 1));
                  wh = lds32(sb + off + tr1 * RB2) >> (8 * (c & 1));
                } else {
                  const int off = o_krc(ri) + (c * NG + gq) * 4;
                  wl = lds32(sb + off + tr0 * RB4);
                  wh = lds32(sb + off + tr1 * RB4);
                }
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                  uint32_t a0, a1, a2, a3;
                  if (two) {
                    a_pairs_2bit(wl, s, a0, a2);
                    a_pairs_2bit(wh, s, a1, a3);
                  } else {
                    a_pairs_4bit(wl, s, a0, a2);
                    a_pairs_4bit(wh, s, a1, a3);
                  }
                  const int fi = (gq * 2 + s) * 32 + lane;
                  if constexpr (MASKB && HL) {   // into the one accumulator: other loops' columns get 0
                    const uint2 bq = QRM[(ri * NG * 2 + gq * 2 + s) * 32 + lane];
                    mma_f16(dsel, a0, a1, a2, a3, bq.x, bq.y);
                  } else if constexpr (MASKB) {
                    const uint4 bq = QRM4[(ri * NG * 2 + gq * 2 + s) * 32 + lane];
                    mma_f16(dsel, a0, a1, a2, a3, bq.x, bq.y);
                    mma_f16(dsel, a0, a1, a2, a3, bq.z, bq.w);
                  } else if constexpr (HL) {
                    const uint2 bq = *reinterpret_cast<const uint2*>((RES4 && !two) ? &QR4[fi] : &QR2[fi]);
                    mma_f16(Dr, a0, a1, a2, a3, bq.x, bq.y);
                  } else {
                    const uint4 bq = (RES4 && !two) ? QR4[fi] : QR2[fi];
                    mma_f16(Dr, a0, a1, a2, a3, bq.x, bq.y);
                    mma_f16(Dr, a0, a1, a2, a3, bq.z, bq.w);
                  }
                }
                // each column keeps its own loop's product
                if constexpr (!MASKB) {
#pragma unroll
                  for (int k = 0; k < 4; ++k) dsel[k] = blend(loop_mask[k & 1][ri], Dr[k], dsel[k]);
                }
              }
            } else {
              // run-time loop count: one accumulator, query fragments masked to each loop's
              // columns
              float Dr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int ri = 0; ri < kMaxResPerBlock; ++ri) {
                if (ri >= nr) break;
                const bool two = !RES4 || a.rbits[ri] == 2;
                uint32_t wl, wh;
                if (two) {
                  const int off = o_krc(ri) + ((c >> 1) * NG + gq) * 4;
                  wl = lds32(sb + off + tr0 * RB2) >> (8 * (c & 1));
                  wh = lds32(sb + off + tr1 * RB2) >> (8 * (c & 1));
                } else {
                  const int off = o_krc(ri) + (c * NG + gq) * 4;
                  wl = lds32(sb + off + tr0 * RB4);
                  wh = lds32(sb + off + tr1 * RB4);
                }
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                  uint32_t a0, a1, a2, a3;
                  if (two) {
                    a_pairs_2bit(wl, s, a0, a2);
                    a_pairs_2bit(wh, s, a1, a3);
                  } else {
                    a_pairs_4bit(wl, s, a0, a2);
                    a_pairs_4bit(wh, s, a1, a3);
                  }
                  const int fi = (gq * 2 + s) * 32 + lane;
                  const uint4 bq = sel4(riB == ri, (RES4 && !two) ? QR4[fi] : QR2[fi]);
                  mma_f16(Dr, a0, a1, a2, a3, bq.x, bq.y);
                  if (!HL) mma_f16(Dr, a0, a1, a2, a3, bq.z, bq.w);
                }
              }
#pragma unroll
              for (int k = 0; k < 4; ++k) dsel[k] = Dr[k];
            }
            // each column's own loop: its step and offset
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float2 m0 = ld_meta(sb + krmD[e] + (tr0 * NG + gq) * 4);
              const float2 m1 = ld_meta(sb + krmD[e] + (tr1 * NG + gq) * 4);
              if constexpr (OFS && PER_LOOP) {   // offsets: above
                E[e] = fmaf(m0.x, dsel[e], E[e]);
                E[2 + e] = fmaf(m1.x, dsel[2 + e], E[2 + e]);
              } else {
                const float qrs = QRsum[gq * NQ + 2 * c + e];
                E[e] = fmaf(m0.x, dsel[e], fmaf(m0.y, qrs, E[e]));
                E[2 + e] = fmaf(m1.x, dsel[2 + e], fmaf(m1.y, qrs, E[2 + e]));
              }
            }
          }
        }
        // score = a_t * reference part + residual part (final loop: the reference alone)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float s_0 = R[e], s_1 = R[2 + e];
          if (nr > 0) {
            const float al0 = ld_half(sb + kaD[e] + tr0 * 2);
            const float al1 = ld_half(sb + kaD[e] + tr1 * 2);
            s_0 = riD[e] >= 0 ? fmaf(al0, s_0, E[e]) : s_0;
            s_1 = riD[e] >= 0 ? fmaf(al1, s_1, E[2 + e]) : s_1;
          }
          if (HL) {   // high part + low part (lanes c and c ^ 2 hold the two)
            s_0 += __shfl_xor_sync(RQ_FULL_MASK, s_0, 2);
            s_1 += __shfl_xor_sync(RQ_FULL_MASK, s_1, 2);
          }
          sc[e] = v0 ? s_0 * code_unit : -INFINITY;
          sc[2 + e] = v1 ? s_1 * code_unit : -INFINITY;
        }
      }

      // ---------------------------------------------------------------- online softmax
      float p[4];
      {
        float tm[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float m = fmaxf(sc[e], sc[2 + e]);
          m = fmaxf(m, __shfl_xor_sync(RQ_FULL_MASK, m, 4));
          m = fmaxf(m, __shfl_xor_sync(RQ_FULL_MASK, m, 8));
          m = fmaxf(m, __shfl_xor_sync(RQ_FULL_MASK, m, 16));
          tm[e] = m;
        }
        const bool n0 = tm[0] > mw[0] + kRescaleSlack, n1 = tm[1] > mw[1] + kRescaleSlack;
        if (__any_sync(RQ_FULL_MASK, n0 || n1)) {
          float corr[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mn = (e ? n1 : n0) ? tm[e] : mw[e];
            corr[e] = (mw[e] == -INFINITY) ? 0.f : exp2f(mw[e] - mn);
            mw[e] = mn;
            lsum[e] *= corr[e];
          }
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              accR[m][k] *= corr[k & 1];
              accE2[m][k] *= corr[k & 1];
              if (RES4) accE4[m][k] *= corr[k & 1];
            }
#pragma unroll
          for (int g = 0; g < (SC ? 1 : NG); ++g)   // (SC: entry 0 holds the lane's two groups)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              offR[g][e] *= corr[e];
              offE[g][e] *= corr[e];
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) p[k] = (sc[k] == -INFINITY) ? 0.f : exp2f(sc[k] - mw[k & 1]);
        lsum[0] += p[0] + p[2];
        lsum[1] += p[1] + p[3];
      }

      // ---------------------------------------------------------------- values
      if constexpr (SC) {
        // weights of tokens tr0, tr1 (the row's lanes all hold its p): p * a for the reference,
        // p for the residual; this lane scales them by the steps of its two groups, and one
        // transpose per token half moves them to the B operand, where column n holds group
        // n & 3 (n >= 4: low parts); each group's MMAs keep their own columns
        float pa0 = p[0], pa1 = p[2], pe0 = 0.f, pe1 = 0.f;
        if (NRT == 1) {
          pe0 = p[0];
          pe1 = p[2];
          if constexpr (MODE == 0) {
            pa0 *= ld_half(sb + vaD[0] + tr0 * 2);
            pa1 *= ld_half(sb + vaD[0] + tr1 * 2);
          }
        }
        uint2 n0 = make_uint2(0u, 0u), n1 = make_uint2(0u, 0u);
        if constexpr (MODE != 2) {
          n0 = *reinterpret_cast<const uint2*>(sb + o_vm + (tr0 * NG + gp) * 4);
          n1 = *reinterpret_cast<const uint2*>(sb + o_vm + (tr1 * NG + gp) * 4);
        }
        if (partial) {   // rows past the context: zero weights and steps whatever the slots hold
          pa0 = v0 ? pa0 : 0.f;
          pa1 = v1 ? pa1 : 0.f;
          pe0 = v0 ? pe0 : 0.f;
          pe1 = v1 ? pe1 : 0.f;
          n0 = v0 ? n0 : make_uint2(0u, 0u);
          n1 = v1 ? n1 : make_uint2(0u, 0u);
        }
        if constexpr (MODE != 2) {   // the reference part
          const float2 u00 = meta_f2(n0.x), u01 = meta_f2(n0.y);
          const float2 u10 = meta_f2(n1.x), u11 = meta_f2(n1.y);
          offR[0][0] = fmaf(pa0, u00.y, fmaf(pa1, u10.y, offR[0][0]));
          offR[0][1] = fmaf(pa0, u01.y, fmaf(pa1, u11.y, offR[0][1]));
          uint32_t b0, b1;
          weights_to_b_packed(pa0 * u00.x, pa0 * u01.x, pa1 * u10.x, pa1 * u11.x, low_lane, b0, b1);
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const bool mine = (r & 3) == g;   // this lane's B column is one of group g's
            const uint32_t g0 = mine ? b0 : 0u, g1 = mine ? b1 : 0u;
            const uint32_t W0 = lds32(sb + o_vc + p0 * D + ((8 * g + r) ^ v_unit_swizzle(p0, D / 4)) * 4);
            const uint32_t W1 = lds32(sb + o_vc + p1 * D + ((8 * g + r) ^ v_unit_swizzle(p1, D / 4)) * 4);
#pragma unroll
            for (int mtg = 0; mtg < 2; ++mtg) {
              uint32_t x0, x1, x2, x3;
              a_pairs_4bit<true>(W0, mtg, x0, x1);
              a_pairs_4bit<true>(W1, mtg, x2, x3);
              mma_f16(accR[2 * g + mtg], x0, x1, x2, x3, g0, g1);
            }
          }
        }
        if (NRT == 1) {
          uint2 q0 = *reinterpret_cast<const uint2*>(sb + vrmD[0] + (tr0 * NG + gp) * 4);
          uint2 q1 = *reinterpret_cast<const uint2*>(sb + vrmD[0] + (tr1 * NG + gp) * 4);
          if (partial) {
            q0 = v0 ? q0 : make_uint2(0u, 0u);
            q1 = v1 ? q1 : make_uint2(0u, 0u);
          }
          const float2 u00 = meta_f2(q0.x), u01 = meta_f2(q0.y);
          const float2 u10 = meta_f2(q1.x), u11 = meta_f2(q1.y);
          offE[0][0] = fmaf(pe0, u00.y, fmaf(pe1, u10.y, offE[0][0]));
          offE[0][1] = fmaf(pe0, u01.y, fmaf(pe1, u11.y, offE[0][1]));
          uint32_t b0, b1;
          weights_to_b_packed(pe0 * u00.x, pe0 * u01.x, pe1 * u10.x, pe1 * u11.x, low_lane, b0, b1);
          const bool two = !RES4 || a.rbits[0] == 2;
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const bool mine = (r & 3) == g;
            const uint32_t g0 = mine ? b0 : 0u, g1 = mine ? b1 : 0u;
            if (two) {
              const int sh = 8 * (r & 1);
              const int u = 4 * g + (r >> 1);
              const uint32_t W0 =
                  lds32(sb + o_vrc(0) + p0 * (2 * RB2) + (u ^ v_unit_swizzle(p0, D / 8)) * 4) >> sh;
              const uint32_t W1 =
                  lds32(sb + o_vrc(0) + p1 * (2 * RB2) + (u ^ v_unit_swizzle(p1, D / 8)) * 4) >> sh;
#pragma unroll
              for (int mtg = 0; mtg < 2; ++mtg) {
                uint32_t x0, x1, x2, x3;
                a_pairs_2bit(W0, mtg, x0, x1);
                a_pairs_2bit(W1, mtg, x2, x3);
                mma_f16(accE2[2 * g + mtg], x0, x1, x2, x3, g0, g1);
              }
            } else if (RES4) {
              const uint32_t W0 =
                  lds32(sb + o_vrc(0) + p0 * D + ((8 * g + r) ^ v_unit_swizzle(p0, D / 4)) * 4);
              const uint32_t W1 =
                  lds32(sb + o_vrc(0) + p1 * D + ((8 * g + r) ^ v_unit_swizzle(p1, D / 4)) * 4);
#pragma unroll
              for (int mtg = 0; mtg < 2; ++mtg) {
                uint32_t x0, x1, x2, x3;
                a_pairs_4bit<true>(W0, mtg, x0, x1);
                a_pairs_4bit<true>(W1, mtg, x2, x3);
                mma_f16(accE4[RES4 ? 2 * g + mtg : 0], x0, x1, x2, x3, g0, g1);
              }
            }
          }
        }
      } else {
        // p * a (reference weights before the step) and p (residual weights before the step)
        // of this lane's score elements; slots past the context may hold any bits
        float pa[4], pe[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float x0 = 1.f, x1 = 1.f;
          if (nr > 0) {
            const float y0 = ld_half(sb + vaD[e] + tr0 * 2);
            const float y1 = ld_half(sb + vaD[e] + tr1 * 2);
            x0 = riD[e] >= 0 ? y0 : 1.f;
            x1 = riD[e] >= 0 ? y1 : 1.f;
          }
          pa[e] = p[e] * x0;
          pa[2 + e] = p[2 + e] * x1;
          pe[e] = riD[e] >= 0 ? p[e] : 0.f;
          pe[2 + e] = riD[e] >= 0 ? p[2 + e] : 0.f;
        }
        uint32_t vm0[NG], vm1[NG];
        load_words<NG>(sb + o_vm + tr0 * NG * 4, vm0);
        load_words<NG>(sb + o_vm + tr1 * NG * 4, vm1);
        if (partial) {   // rows past the context: zero weights and steps whatever the slots hold
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            pa[e] = v0 ? pa[e] : 0.f;
            pa[2 + e] = v1 ? pa[2 + e] : 0.f;
            pe[e] = v0 ? pe[e] : 0.f;
            pe[2 + e] = v1 ? pe[2 + e] : 0.f;
          }
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            vm0[g] = v0 ? vm0[g] : 0u;
            vm1[g] = v1 ? vm1[g] : 0u;
          }
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float2 m0 = meta_f2(vm0[g]), m1 = meta_f2(vm1[g]);
          offR[g][0] = fmaf(pa[0], m0.y, fmaf(pa[2], m1.y, offR[g][0]));
          offR[g][1] = fmaf(pa[1], m0.y, fmaf(pa[3], m1.y, offR[g][1]));
          uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
          if constexpr (HL)
            weights_to_b_packed(pa[0] * m0.x, pa[1] * m0.x, pa[2] * m1.x, pa[3] * m1.x, low_lane,
                                bh0, bh1);
          else
            weights_to_b(pa[0] * m0.x, pa[1] * m0.x, pa[2] * m1.x, pa[3] * m1.x, bh0, bh1, bl0, bl1);
          const uint32_t W0 = lds32(sb + o_vc + p0 * D + ((8 * g + r) ^ v_unit_swizzle(p0, D / 4)) * 4);
          const uint32_t W1 = lds32(sb + o_vc + p1 * D + ((8 * g + r) ^ v_unit_swizzle(p1, D / 4)) * 4);
#pragma unroll
          for (int mtg = 0; mtg < 2; ++mtg) {
            uint32_t x0, x1, x2, x3;
            a_pairs_4bit<true>(W0, mtg, x0, x1);
            a_pairs_4bit<true>(W1, mtg, x2, x3);
            mma_f16(accR[2 * g + mtg], x0, x1, x2, x3, bh0, bh1);
            if (!HL) mma_f16(accR[2 * g + mtg], x0, x1, x2, x3, bl0, bl1);
          }
        }
        if (nr > 0) {
          // each D column's own loop: its value step and offset, tokens tr0 and tr1
          uint32_t rm0[2][NG], rm1[2][NG];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            load_words<NG>(sb + vrmD[e] + tr0 * NG * 4, rm0[e]);
            load_words<NG>(sb + vrmD[e] + tr1 * NG * 4, rm1[e]);
            if (partial) {
#pragma unroll
              for (int g = 0; g < NG; ++g) {
                rm0[e][g] = v0 ? rm0[e][g] : 0u;
                rm1[e][g] = v1 ? rm1[e][g] : 0u;
              }
            }
          }
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            float w[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float2 m0 = meta_f2(rm0[e][g]), m1 = meta_f2(rm1[e][g]);
              w[e] = pe[e] * m0.x;
              w[2 + e] = pe[2 + e] * m1.x;
              offE[g][e] = fmaf(pe[e], m0.y, fmaf(pe[2 + e], m1.y, offE[g][e]));
            }
            uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
            if constexpr (HL)
              weights_to_b_packed(w[0], w[1], w[2], w[3], low_lane, bh0, bh1);
            else
              weights_to_b(w[0], w[1], w[2], w[3], bh0, bh1, bl0, bl1);
#pragma unroll
            for (int ri = 0; ri < kMaxResPerBlock; ++ri) {
              if (ri >= nr) break;
              // weights of the other loops' columns are masked (one loop: nothing to mask)
              const bool keep = (NRT == 1) || (riB == ri);
              const uint32_t eh0 = keep ? bh0 : 0u, eh1 = keep ? bh1 : 0u;
              const uint32_t el0 = keep ? bl0 : 0u, el1 = keep ? bl1 : 0u;
              if (!RES4 || a.rbits[ri] == 2) {
                const int sh = 8 * (r & 1);
                const int u = 4 * g + (r >> 1);
                const uint32_t W0 =
                    lds32(sb + o_vrc(ri) + p0 * (2 * RB2) + (u ^ v_unit_swizzle(p0, D / 8)) * 4) >> sh;
                const uint32_t W1 =
                    lds32(sb + o_vrc(ri) + p1 * (2 * RB2) + (u ^ v_unit_swizzle(p1, D / 8)) * 4) >> sh;
#pragma unroll
                for (int mtg = 0; mtg < 2; ++mtg) {
                  uint32_t x0, x1, x2, x3;
                  a_pairs_2bit(W0, mtg, x0, x1);
                  a_pairs_2bit(W1, mtg, x2, x3);
                  mma_f16(accE2[2 * g + mtg], x0, x1, x2, x3, eh0, eh1);
                  if (!HL) mma_f16(accE2[2 * g + mtg], x0, x1, x2, x3, el0, el1);
                }
              } else if (RES4) {
                const uint32_t W0 =
                    lds32(sb + o_vrc(ri) + p0 * D + ((8 * g + r) ^ v_unit_swizzle(p0, D / 4)) * 4);
                const uint32_t W1 =
                    lds32(sb + o_vrc(ri) + p1 * D + ((8 * g + r) ^ v_unit_swizzle(p1, D / 4)) * 4);
#pragma unroll
                for (int mtg = 0; mtg < 2; ++mtg) {
                  uint32_t x0, x1, x2, x3;
                  a_pairs_4bit<true>(W0, mtg, x0, x1);
                  a_pairs_4bit<true>(W1, mtg, x2, x3);
                  mma_f16(accE4[RES4 ? 2 * g + mtg : 0], x0, x1, x2, x3, eh0, eh1);
                  if (!HL) mma_f16(accE4[RES4 ? 2 * g + mtg : 0], x0, x1, x2, x3, el0, el1);
                }
              }
            }
          }
        }
      }
    }
    // this warp is done with the stage; the last of the four refills it
    __syncwarp();
    if (lane == 0) {
      if (atom_add_acq_rel(&cnt[st], 1u) == unsigned(kW - 1)) {
        cnt[st] = 0u;
        if (i + S < ntiles) {
          fence_proxy_async_smem();
          issue(i + S);
          cnt[kIssuedSlot] = unsigned(i + S + 1);
        }
      }
    }
  }

  if (__syncthreads_or(failed)) {
    // a copy never completed: flag it, wait (bounded) for the copies still in flight, and
    // take the ticket without records (the combine's output is NaN)
    if (threadIdx.x == 0) {
      atomicOr(a.err, 1u);
      const int issued = int(cnt[kIssuedSlot]);
      for (int t = issued - S < 0 ? 0 : issued - S; t < issued; ++t)
        mbar_wait_bounded(smem_u32(&bars[t % S]), uint32_t((t / S) & 1), a.wait_limit_ns);
    }
    combine_if_last();
    return;
  }

  // ------------------------------------------------------------------ merge the four warps
  // every issued copy has landed and been consumed: the stage memory is free
  // softmax sums and value offsets: over the 8 row lanes (tokens)
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float v = lsum[e];
    v += __shfl_xor_sync(RQ_FULL_MASK, v, 4);
    v += __shfl_xor_sync(RQ_FULL_MASK, v, 8);
    v += __shfl_xor_sync(RQ_FULL_MASK, v, 16);
    lsum[e] = v;
#pragma unroll
    for (int g = 0; g < (SC ? 1 : NG); ++g) {
      float x = offR[g][e], y = offE[g][e];
      x += __shfl_xor_sync(RQ_FULL_MASK, x, 4);
      y += __shfl_xor_sync(RQ_FULL_MASK, y, 4);
      x += __shfl_xor_sync(RQ_FULL_MASK, x, 8);
      y += __shfl_xor_sync(RQ_FULL_MASK, y, 8);
      x += __shfl_xor_sync(RQ_FULL_MASK, x, 16);
      y += __shfl_xor_sync(RQ_FULL_MASK, y, 16);
      offR[g][e] = x;
      offE[g][e] = y;
    }
  }
  if (r == 0) {
    red[warp * NQ + 2 * c] = mw[0];
    red[warp * NQ + 2 * c + 1] = mw[1];
  }
  __syncthreads();
  float f[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float M = red[2 * c + e];
#pragma unroll
    for (int w = 1; w < kW; ++w) M = fmaxf(M, red[w * NQ + 2 * c + e]);
    f[e] = (mw[e] == -INFINITY) ? 0.f : exp2f(mw[e] - M);
  }
  if (r == 0) {
    red[kW * NQ + warp * NQ + 2 * c] = lsum[0] * f[0];
    red[kW * NQ + warp * NQ + 2 * c + 1] = lsum[1] * f[1];
  }
  if (HL) {   // accumulator columns 4-7 hold the low-part products of columns 0-3
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        accR[m][k] += __shfl_xor_sync(RQ_FULL_MASK, accR[m][k], 2);
        accE2[m][k] += __shfl_xor_sync(RQ_FULL_MASK, accE2[m][k], 2);
        if (RES4) accE4[m][k] += __shfl_xor_sync(RQ_FULL_MASK, accE4[m][k], 2);
      }
  }
  // this warp's rescaled partial accumulators: buf[warp][column][acc_ref D | acc_res D], rows
  // padded by 4 floats so that the float4 stores of a quarter-warp hit distinct banks (query
  // columns of the block only)
  constexpr int BS = 2 * D + 4;
  float* buf = reinterpret_cast<float*>(smem);
  if constexpr (SC) {
    // the block's one column: group g (channels 32 g ..) sits in lane column c = g / 2,
    // element e = g % 2, high and low parts added above
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      if ((g >> 1) != c) continue;
      const int e = g & 1;
      float* o = buf + (warp * NQ) * BS;
      float vr[4], ve[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int mtg = j >> 1, hh = j & 1, k = 2 * hh + e;
        const float sc4 = hh ? 0.0625f : 1.f;
        const float sc2 = 16777216.f / float(1 << (2 * j));   // 2-bit codes: subnormal
        vr[j] = fmaf(accR[2 * g + mtg][k], sc4, offR[0][e]) * f[e];
        float x = fmaf(accE2[2 * g + mtg][k], sc2, offE[0][e]);
        if (RES4) x = fmaf(accE4[RES4 ? 2 * g + mtg : 0][k], sc4, x);
        ve[j] = x * f[e];
      }
      *reinterpret_cast<float4*>(o + 32 * g + 4 * r) = make_float4(vr[0], vr[1], vr[2], vr[3]);
      *reinterpret_cast<float4*>(o + D + 32 * g + 4 * r) = make_float4(ve[0], ve[1], ve[2], ve[3]);
    }
  }
#pragma unroll
  for (int e = 0; e < 2 && !SC; ++e) {
    const int n = 2 * c + e;
    if (!(n / blk.gw < blk.nl && blk.gi0 + n % blk.gw < a.g)) continue;
    float* o = buf + (warp * NQ + n) * BS;
    // channels 32 g + 4 r + j of column n, j = 2 mtg + hh (hh: fragment row r or r + 8)
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float vr[4], ve[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int mtg = j >> 1, hh = j & 1, k = 2 * hh + e;
        const float sc4 = hh ? 0.0625f : 1.f;     // value codes are normal fp16
        const float sc2 = 16777216.f / float(1 << (2 * j));   // 2-bit codes: subnormal
        vr[j] = fmaf(accR[2 * g + mtg][k], sc4, offR[g][e]) * f[e];
        float x = fmaf(accE2[2 * g + mtg][k], sc2, offE[g][e]);
        if (RES4) x = fmaf(accE4[RES4 ? 2 * g + mtg : 0][k], sc4, x);
        ve[j] = x * f[e];
      }
      *reinterpret_cast<float4*>(o + 32 * g + 4 * r) = make_float4(vr[0], vr[1], vr[2], vr[3]);
      *reinterpret_cast<float4*>(o + D + 32 * g + 4 * r) = make_float4(ve[0], ve[1], ve[2], ve[3]);
    }
  }
  __syncthreads();
  const int rec = int(partial_floats_d(D));
  auto rec_ptr = [&](int col) -> float* {
    const int li = col / blk.gw, gi = blk.gi0 + col % blk.gw;
    if (li >= blk.nl || gi >= a.g) return nullptr;
    const int lc = blk.lb + li - a.loop_begin;
    const int64_t hq = int64_t(h) * a.g + gi;
    return a.part + (((int64_t(b) * a.Hq + hq) * a.loop_count + lc) * a.n_splits + split) * rec;
  };
  if (threadIdx.x < NQ) {
    float* o = rec_ptr(threadIdx.x);
    if (o) {
      float M = red[threadIdx.x], ls = 0.f;
#pragma unroll
      for (int w = 1; w < kW; ++w) M = fmaxf(M, red[w * NQ + threadIdx.x]);
#pragma unroll
      for (int w = 0; w < kW; ++w) ls += red[kW * NQ + w * NQ + threadIdx.x];
      o[0] = M;
      o[1] = ls;
    }
  }
  // records: m, l, 2 pad, acc_ref, acc_res (16-byte aligned)
  for (int idx = threadIdx.x; idx < NQ * (D / 2); idx += kW * 32) {
    const int col = idx / (D / 2), q4 = idx % (D / 2);
    float* o = rec_ptr(col);
    if (!o) continue;
    float4 v = *reinterpret_cast<const float4*>(buf + col * BS + 4 * q4);
#pragma unroll
    for (int w = 1; w < kW; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(buf + (w * NQ + col) * BS + 4 * q4);
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    *reinterpret_cast<float4*>(o + 4 + 4 * q4) = v;
  }
  combine_if_last();
}

}  // namespace

// Single-column packing exists for head dim 128 and one loop (the final one, or one residual
// loop of 2 or 4 bits).
inline bool has_single_column_variant(int D, bool res4, int nr) {
  return D == 128 && (res4 ? nr == 1 : nr <= 1);
}

namespace {

template <int D, bool PG, int PK>
KernelFn pick_generic(bool res4) {
  return res4 ? rq_mma_kernel<D, true, -1, PG, PK> : rq_mma_kernel<D, false, -1, PG, PK>;
}

// Variants with the residual-loop count fixed at compile time, for the common blocks: one
// loop of a per-loop call (0 or 1 residual), two loops of a 4-query-head GQA block (2) and
// all four loops of a 4-loop model (3); each for a contiguous and for a paged cache and for
// each packing of the MMA columns.  Single-column packing exists for head dim 128 and one
// loop; other blocks given it take the 4-column packing.
template <bool PG, int PK>
KernelFn pick_pg(int D, bool res4, int nr) {
  if constexpr (PK == 2) {
    if (has_single_column_variant(D, res4, nr))
      return nr == 0 ? rq_mma_kernel<128, false, 0, PG, 2>
                     : (res4 ? rq_mma_kernel<128, true, 1, PG, 2> : rq_mma_kernel<128, false, 1, PG, 2>);
    return pick_pg<PG, 1>(D, res4, nr);
  } else {
    if (D == 128 && !res4) {
      if (nr == 0) return rq_mma_kernel<128, false, 0, PG, PK>;
      if (nr == 1) return rq_mma_kernel<128, false, 1, PG, PK>;
      if (nr == 2) return rq_mma_kernel<128, false, 2, PG, PK>;
      if (nr == 3) return rq_mma_kernel<128, false, 3, PG, PK>;
    }
    if (D == 128 && res4) {
      if (nr == 1) return rq_mma_kernel<128, true, 1, PG, PK>;
      if (nr == 3) return rq_mma_kernel<128, true, 3, PG, PK>;
    }
    if (D == 64 && !res4) {
      if (nr == 0) return rq_mma_kernel<64, false, 0, PG, PK>;
      if (nr == 1) return rq_mma_kernel<64, false, 1, PG, PK>;
      if (nr == 3) return rq_mma_kernel<64, false, 3, PG, PK>;
    }
    return D == 128 ? pick_generic<128, PG, PK>(res4) : pick_generic<64, PG, PK>(res4);
  }
}

}  // namespace

// kernel of the paged-cache variants (rq_decode_mma_paged.cu)
KernelFn pick_paged(int D, bool res4, int nr, int pk);

}  // namespace rq
