// ResidualQuant split-KV decode attention on the tensor cores (sm_103a).
//
// Per CTA: one (split of the context, kv-head, sequence); 4 warps; 64-token tiles of every
// packed array are staged in shared memory by 1-D bulk (TMA) copies through a multi-stage
// mbarrier pipeline.  For a loop-l query q and token t (rit.work summary, "How each pass's
// KV cache is reconstructed": reference and residuals rebuilt inside attention)
//   score_t = a_t * sum_g [s^r_g,t (q_g . c^r_g,t) + z^r_g,t sum(q_g)]
//           +       sum_g [s^e_g,t (q'_g . c^e_g,t) + z^e_g,t sum(q'_g)],      q' = R q
//   acc_ref += p_t a_t (s^r c^r + z^r),   acc_res += p_t (s^e c^e + z^e)   (rotated domain)
// The code dot products and the P.V products run as mma.sync m16n8k16 (f16 in, f32 acc):
//   scores: M = 16 tokens, N = 8 query columns, K = 16 channels of one 32-channel group;
//   values: M = 16 channels of one group, N = 8 query columns, K = 16 tokens.
// A pair of packed codes becomes an f16x2 operand with one AND: the code bits, masked in
// place with a zero exponent field, are the fp16 subnormal c * 2^-24 times a power of two
// fixed by their bit position; that power is folded into the query fragments (scores) or
// removed per output row at the end (values), and 2^24 is restored in fp32.  The other operand (queries, softmax weights) is split into an fp16 high part
// and an fp16 low part (two MMAs) and so carries about 22 significant bits; products are
// exact in the fp32 accumulators.
// Query columns of every loop share the fragments: the residual codes of loop l meet a
// query fragment whose columns of other loops are masked to zero, so all residual loops
// accumulate into one score fragment per group (scaled once by each column's own step and
// offset) and into one value accumulator per residual bit width.
#include <mutex>

#include "rq_common.cuh"
#include "rq_kernels.h"
#include "rq_ptx.cuh"

namespace rq {
namespace {

constexpr int kT = 64;                        // tokens per tile
constexpr int kW = 4;                         // warps per CTA
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct MmaArgs {
  const uint8_t* kc;
  const uint16_t* km;
  const uint8_t* vc;
  const uint16_t* vm;
  const uint8_t* krc[kMaxResPerBlock];
  const uint16_t* krm[kMaxResPerBlock];
  const uint16_t* ka[kMaxResPerBlock];
  const uint8_t* vrc[kMaxResPerBlock];
  const uint16_t* vrm[kMaxResPerBlock];
  const uint16_t* va[kMaxResPerBlock];
  int rbits[kMaxResPerBlock];
  const int8_t* ksigns;
  const uint16_t* q;
  const int32_t* ctx_lens;
  float* part;
  unsigned* err;
  int B, Hq, H, L, cap, g, loop_begin, loop_count, n_splits, tokens_per_split;
  QueryBlock blk;
  float scale_log2;
  int n_stages, stage_bytes;
  int off_kc, off_km, off_vc, off_vm;
  int off_krc[kMaxResPerBlock], off_krm[kMaxResPerBlock], off_ka[kMaxResPerBlock];
  int off_vrc[kMaxResPerBlock], off_vrm[kMaxResPerBlock], off_va[kMaxResPerBlock];
};

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

__device__ __forceinline__ uint4 sel4(bool keep, uint4 v) {
  return keep ? v : make_uint4(0u, 0u, 0u, 0u);
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

// NRT >= 0: the block's number of residual loops, fixed at compile time; -1: read at run time.
template <int D, int NT, bool RES4, int NRT>
__global__ void __launch_bounds__(kW * 32) rq_mma_kernel(const __grid_constant__ MmaArgs a) {
  constexpr int NG = D / 32;
  constexpr int NQP = NT * 8;        // query columns (padded)
  constexpr int P = D / 32;          // channels per lane in the query prep
  constexpr int RB4 = D / 2;         // bytes of a 4-bit row
  constexpr int RB2 = D / 4;         // bytes of a 2-bit row
  constexpr int MTW = (D == 128) ? 2 : 1;  // 16-channel M-tiles per warp in the value phase
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const QueryBlock blk = a.blk;
  const int nr = NRT >= 0 ? NRT : blk.nr;

  const SmemLayout lay = smem_layout(D, NT, RES4, a.n_stages, a.stage_bytes);
  const int PR = lay.prow;
  uint4* QF = reinterpret_cast<uint4*>(smem + lay.qf);
  uint4* QR2 = reinterpret_cast<uint4*>(smem + lay.qr2);
  uint4* QR4 = reinterpret_cast<uint4*>(smem + lay.qr4);
  float* Qsum = reinterpret_cast<float*>(smem + lay.qsum);
  float* QRsum = reinterpret_cast<float*>(smem + lay.qrsum);
  float* Ps = reinterpret_cast<float*>(smem + lay.ps);
  float* Pa = reinterpret_cast<float*>(smem + lay.pa);
  float* red = reinterpret_cast<float*>(smem + lay.red);
  float* mrun = reinterpret_cast<float*>(smem + lay.mrun);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);

  // residual index (into the block's residual loops) of query column n, -1 if the column
  // is the final loop's or a padding column
  auto col_ri = [&](int n) -> int {
    const int li = n / blk.gw, gi = blk.gi0 + n % blk.gw;
    const int l = blk.lb + li;
    return (li < blk.nl && gi < a.g && l != a.L - 1) ? l - blk.r0 : -1;
  };

  // ------------------------------------------------------------------ query preparation
  {
    uint32_t* z32 = reinterpret_cast<uint32_t*>(smem + lay.qf);
    const int nz = (lay.mrun - lay.qf) / 4;
    for (int i = threadIdx.x; i < nz; i += blockDim.x) z32[i] = 0u;
    for (int i = threadIdx.x; i < NQP; i += blockDim.x) mrun[i] = -INFINITY;
  }
  __syncthreads();
  // query columns of this block: scaled q, rotated q' = R q, per-group sums
  auto prep_column = [&](int n, float (&v)[P], float (&rr)[P]) -> bool {
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
    return real;
  };
  // pass 1: the largest |q|, |q'| of the block fixes a power-of-two fragment scale 2^k with
  // max |fragment| <= 2^14, so the low parts of the split stay normal fp16 (they meet the
  // subnormal code operands of the score MMAs)
  {
    float mx = 0.f;
    for (int n = warp; n < NQP; n += kW) {
      float v[P], rr[P];
      prep_column(n, v, rr);
#pragma unroll
      for (int j = 0; j < P; ++j) mx = fmaxf(mx, fmaxf(fabsf(v[j]), fabsf(rr[j])));
    }
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
  __syncthreads();
  if (threadIdx.x == 0) *reinterpret_cast<unsigned*>(red) = 0u;
  // pass 2: fragments and group sums
  for (int n = warp; n < NQP; n += kW) {
    float v[P], rr[P];
    const bool real = prep_column(n, v, rr);
    (void)real;
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
    if ((lane & (32 / P - 1)) == 0) {
      Qsum[grp * NQP + n] = s1;
      if (ri >= 0) QRsum[grp * NQP + n] = s2;
    }
    const int nt = n >> 3, nn = n & 7;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const int ch = lane * P + j, gq = ch >> 5, cl = ch & 31;
      const float vq = v[j] * qscale, rq = rr[j] * qscale;
      {  // 4-bit mapping: slot (c4, s, hi, e) <- channel 8 c4 + 2 s + hi + 4 e, scale 16^-hi
        const int c4 = cl >> 3, w8 = cl & 7, s = (w8 >> 1) & 1, hi = w8 & 1, e = w8 >> 2;
        const int idx = ((gq * 2 + s) * NT + nt) * 32 + nn * 4 + c4;
        __half* dq = reinterpret_cast<__half*>(&QF[idx]);
        split_half(hi ? vq * 0.0625f : vq, dq[hi * 2 + e], dq[4 + hi * 2 + e]);
        if (RES4 && bits == 4) {
          __half* dr = reinterpret_cast<__half*>(&QR4[idx]);
          split_half(hi ? rq * 0.0625f : rq, dr[hi * 2 + e], dr[4 + hi * 2 + e]);
        }
      }
      if (bits == 2) {  // 2-bit mapping: slot (cq, s, hi, e) <- channel 16(cq/2)+4(cq%2)+2s+hi+8e
        const int e = (cl >> 3) & 1, cq = 2 * (cl >> 4) + ((cl & 7) >> 2), jj = cl & 3;
        const int s = jj >> 1, hi = jj & 1;
        const float sc = (jj == 0) ? 1.f : (jj == 1) ? 0.25f : (jj == 2) ? 0.0625f : 0.015625f;
        __half* dr = reinterpret_cast<__half*>(&QR2[((gq * 2 + s) * NT + nt) * 32 + nn * 4 + cq]);
        split_half(rq * sc, dr[hi * 2 + e], dr[4 + hi * 2 + e]);
      }
    }
  }

  // ------------------------------------------------------------------ pipeline set-up
  const int ctx = min(a.ctx_lens[b], a.cap);
  const int t_begin = split * a.tokens_per_split;
  const int t_end = min(ctx, t_begin + a.tokens_per_split);
  const int ntiles = t_end > t_begin ? (t_end - t_begin + kT - 1) / kT : 0;
  const int64_t slot = int64_t(b) * a.H + h;
  const int S = a.n_stages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto issue = [&](int tile) {
    const int st = tile % S;
    const uint32_t bar = smem_u32(&bars[st]);
    const uint32_t dst = smem_u32(smem + st * a.stage_bytes);
    const int64_t tok = slot * a.cap + t_begin + int64_t(tile) * kT;
    mbar_arrive_expect_tx(bar, uint32_t(a.stage_bytes));
    bulk_g2s(dst + a.off_kc, a.kc + tok * RB4, kT * RB4, bar);
    bulk_g2s(dst + a.off_km, a.km + tok * NG * 2, kT * NG * 4, bar);
    bulk_g2s(dst + a.off_vc, a.vc + tok * RB4, kT * RB4, bar);
    bulk_g2s(dst + a.off_vm, a.vm + tok * NG * 2, kT * NG * 4, bar);
#pragma unroll
    for (int ri = 0; ri < kMaxResPerBlock; ++ri) {
      if (ri >= nr) break;
      const int rb = D * a.rbits[ri] / 8;
      bulk_g2s(dst + a.off_krc[ri], a.krc[ri] + tok * rb, kT * rb, bar);
      bulk_g2s(dst + a.off_krm[ri], a.krm[ri] + tok * NG * 2, kT * NG * 4, bar);
      bulk_g2s(dst + a.off_ka[ri], a.ka[ri] + tok, kT * 2, bar);
      bulk_g2s(dst + a.off_vrc[ri], a.vrc[ri] + tok * rb, kT * rb, bar);
      bulk_g2s(dst + a.off_vrm[ri], a.vrm[ri] + tok * NG * 2, kT * NG * 4, bar);
      bulk_g2s(dst + a.off_va[ri], a.va[ri] + tok, kT * 2, bar);
    }
  };
  int next_issue = 0;  // tiles issued so far (thread 0)
  if (threadIdx.x == 0) {
    for (; next_issue < S && next_issue < ntiles; ++next_issue) issue(next_issue);
  }

  // residual indices of this lane's B-fragment columns (nt*8 + r) and D-fragment columns
  // (nt*8 + 2c + e)
  int riB[NT], riD[NT][2];
  int krmD[NT][2], kaD[NT][2], vaD[NT][2], vrmB[NT];   // stage offsets of those columns' loops
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    riB[nt] = col_ri(nt * 8 + r);
    vrmB[nt] = pick_int(a.off_vrm, riB[nt] < 0 ? 0 : riB[nt]);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      riD[nt][e] = col_ri(nt * 8 + 2 * c + e);
      const int rc = riD[nt][e] < 0 ? 0 : riD[nt][e];
      krmD[nt][e] = pick_int(a.off_krm, rc);
      kaD[nt][e] = pick_int(a.off_ka, rc);
      vaD[nt][e] = pick_int(a.off_va, rc);
    }
  }

  float lpart[NT][2];
  float accR[MTW][NT][4], accE2[MTW][NT][4], accE4[RES4 ? MTW : 1][NT][4];
  float offR[NT], offE[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    lpart[nt][0] = lpart[nt][1] = 0.f;
    offR[nt] = offE[nt] = 0.f;
#pragma unroll
    for (int m = 0; m < MTW; ++m)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        accR[m][nt][k] = 0.f;
        accE2[m][nt][k] = 0.f;
        if (RES4) accE4[m][nt][k] = 0.f;
      }
  }
  const int gv = (D == 128) ? warp : (warp >> 1);     // value-phase channel group of this warp

  bool failed = false;
  int fail_tile = 0;
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % S;
    const bool ok = mbar_wait_bounded(smem_u32(&bars[st]), uint32_t((i / S) & 1), kWaitLimitNs);
    const uint8_t* sb = smem + st * a.stage_bytes;
    const int t0 = t_begin + i * kT;

    // -------------------------------------------------------------- scores (16 tokens/warp)
    const int tr0 = 16 * warp + r, tr1 = tr0 + 8;
    const bool v0 = t0 + tr0 < t_end, v1 = t0 + tr1 < t_end;
    float sc[NT][4];
    {
      float Sref[NT][4], Sres[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) Sref[nt][k] = Sres[nt][k] = 0.f;
      float2 mk0[NG], mk1[NG];
#pragma unroll
      for (int gq = 0; gq < NG; ++gq) {
        mk0[gq] = ld_meta(sb + a.off_km + (tr0 * NG + gq) * 4);
        mk1[gq] = ld_meta(sb + a.off_km + (tr1 * NG + gq) * 4);
      }
      // this lane's word of every group (K rows are group-interleaved: one load)
      uint32_t kw0[NG], kw1[NG];
      load_words<NG>(sb + a.off_kc + tr0 * RB4 + c * NG * 4, kw0);
      load_words<NG>(sb + a.off_kc + tr1 * RB4 + c * NG * 4, kw1);
#pragma unroll
      for (int gq = 0; gq < NG; ++gq) {
        // reference
        {
          const uint32_t wl = kw0[gq];
          const uint32_t wh = kw1[gq];
          float Dg[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) Dg[nt][k] = 0.f;
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            uint32_t a0, a2, a1, a3;
            a_pairs_4bit(wl, s, a0, a2);
            a_pairs_4bit(wh, s, a1, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint4 bq = QF[((gq * 2 + s) * NT + nt) * 32 + lane];
              mma_f16(Dg[nt], a0, a1, a2, a3, bq.x, bq.y);
              mma_f16(Dg[nt], a0, a1, a2, a3, bq.z, bq.w);
            }
          }
          const float s0 = mk0[gq].x * code_unit, s1 = mk1[gq].x * code_unit;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float2 qs = *reinterpret_cast<const float2*>(&Qsum[gq * NQP + nt * 8 + 2 * c]);
            Sref[nt][0] += s0 * Dg[nt][0] + mk0[gq].y * qs.x;
            Sref[nt][1] += s0 * Dg[nt][1] + mk0[gq].y * qs.y;
            Sref[nt][2] += s1 * Dg[nt][2] + mk1[gq].y * qs.x;
            Sref[nt][3] += s1 * Dg[nt][3] + mk1[gq].y * qs.y;
          }
        }
        // residuals of every loop of the block, one fragment
        if (nr > 0) {
          float Dr[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) Dr[nt][k] = 0.f;
#pragma unroll
          for (int ri = 0; ri < kMaxResPerBlock; ++ri) {
            if (ri >= nr) break;
            const int nt_ri = ((blk.r0 + ri - blk.lb) * blk.gw) >> 3;
            const bool two = a.rbits[ri] == 2;
            uint32_t wl, wh;
            if (two) {
              const int off = a.off_krc[ri] + ((c >> 1) * NG + gq) * 4;
              wl = lds32(sb + off + tr0 * RB2) >> (8 * (c & 1));
              wh = lds32(sb + off + tr1 * RB2) >> (8 * (c & 1));
            } else {
              const int off = a.off_krc[ri] + (c * NG + gq) * 4;
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
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt != nt_ri) continue;
                const int fi = ((gq * 2 + s) * NT + nt) * 32 + lane;
                const uint4 bq = sel4(riB[nt] == ri, (RES4 && !two) ? QR4[fi] : QR2[fi]);
                mma_f16(Dr[nt], a0, a1, a2, a3, bq.x, bq.y);
                mma_f16(Dr[nt], a0, a1, a2, a3, bq.z, bq.w);
              }
            }
          }
          // each column's own loop: its step and offset
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int ri = riD[nt][e];
              const float2 m0 = ld_meta(sb + krmD[nt][e] + (tr0 * NG + gq) * 4);
              const float2 m1 = ld_meta(sb + krmD[nt][e] + (tr1 * NG + gq) * 4);
              const float qrs = QRsum[gq * NQP + nt * 8 + 2 * c + e];
              const float d0 = (m0.x * code_unit) * Dr[nt][e] + m0.y * qrs;
              const float d1 = (m1.x * code_unit) * Dr[nt][2 + e] + m1.y * qrs;
              Sres[nt][e] += ri >= 0 ? d0 : 0.f;
              Sres[nt][2 + e] += ri >= 0 ? d1 : 0.f;
            }
          }
        }
      }
      // score = a_t * reference part + residual part (final loop: the reference alone)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ri = riD[nt][e];
          float s_0 = Sref[nt][e], s_1 = Sref[nt][2 + e];
          if (nr > 0) {
            const float al0 = ld_half(sb + kaD[nt][e] + tr0 * 2);
            const float al1 = ld_half(sb + kaD[nt][e] + tr1 * 2);
            s_0 = ri >= 0 ? al0 * s_0 + Sres[nt][e] : s_0;
            s_1 = ri >= 0 ? al1 * s_1 + Sres[nt][2 + e] : s_1;
          }
          sc[nt][e] = v0 ? s_0 : -INFINITY;
          sc[nt][2 + e] = v1 ? s_1 : -INFINITY;
        }
      }
    }
    // per-warp column maxima over its 16 tokens
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float m0 = fmaxf(sc[nt][0], sc[nt][2]), m1 = fmaxf(sc[nt][1], sc[nt][3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(RQ_FULL_MASK, m0, o));
        m1 = fmaxf(m1, __shfl_xor_sync(RQ_FULL_MASK, m1, o));
      }
      if (r == 0) {
        red[warp * NQP + nt * 8 + 2 * c] = m0;
        red[warp * NQP + nt * 8 + 2 * c + 1] = m1;
      }
    }
    if (__syncthreads_or(!ok)) {  // (A)
      failed = true;
      fail_tile = i;
      break;
    }
    // ---------------------------------------------------------------- online softmax
    float corr[NT][2];
    float mnew_mine = 0.f;
    if (threadIdx.x < NQP) {
      float mt = red[threadIdx.x];
#pragma unroll
      for (int w = 1; w < kW; ++w) mt = fmaxf(mt, red[w * NQP + threadIdx.x]);
      mnew_mine = fmaxf(mrun[threadIdx.x], mt);
    }
    // value-offset sums are kept per B-fragment column nt*8 + r
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = nt * 8 + r;
      float mt = red[col];
#pragma unroll
      for (int w = 1; w < kW; ++w) mt = fmaxf(mt, red[w * NQP + col]);
      const float mo = mrun[col];
      const float cb = (mo == -INFINITY) ? 0.f : exp2f(mo - fmaxf(mo, mt));
      offR[nt] *= cb;
      offE[nt] *= cb;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = nt * 8 + 2 * c + e;
        float mt = red[col];
#pragma unroll
        for (int w = 1; w < kW; ++w) mt = fmaxf(mt, red[w * NQP + col]);
        const float mo = mrun[col];
        const float mn = fmaxf(mo, mt);
        corr[nt][e] = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
        const float p0 = exp2f(sc[nt][e] - mn), p1 = exp2f(sc[nt][2 + e] - mn);
        lpart[nt][e] = lpart[nt][e] * corr[nt][e] + p0 + p1;
        const int ri = riD[nt][e];
        float a0v = 1.f, a1v = 1.f;
        if (nr > 0) {
          const float x0 = ld_half(sb + vaD[nt][e] + tr0 * 2);
          const float x1 = ld_half(sb + vaD[nt][e] + tr1 * 2);
          a0v = ri >= 0 ? x0 : 1.f;
          a1v = ri >= 0 ? x1 : 1.f;
        }
        Ps[tr0 * PR + col] = v0 ? p0 : 0.f;
        Ps[tr1 * PR + col] = v1 ? p1 : 0.f;
        Pa[tr0 * PR + col] = v0 ? p0 * a0v : 0.f;
        Pa[tr1 * PR + col] = v1 ? p1 * a1v : 0.f;
      }
    }
    // the stage read by tile i-1 is free (every warp is past barrier A): refill it
    if (threadIdx.x == 0 && i >= 1 && i + S - 1 < ntiles) {
      issue(i + S - 1);
      next_issue = i + S;
    }
    __syncthreads();  // (B)
    if (threadIdx.x < NQP) mrun[threadIdx.x] = mnew_mine;

    // ------------------------------------------------------------ values (one group/warp)
#pragma unroll
    for (int m = 0; m < MTW; ++m)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          accR[m][nt][k] *= corr[nt][k & 1];
          accE2[m][nt][k] *= corr[nt][k & 1];
          if (RES4) accE4[m][nt][k] *= corr[nt][k & 1];
        }
#pragma unroll
    for (int ks = 0; ks < kT / 16; ++ks) {
      int tt[4];
      tt[0] = 16 * ks + 2 * c;
      tt[1] = tt[0] + 1;
      tt[2] = tt[0] + 8;
      tt[3] = tt[0] + 9;
      const int p0 = 8 * ks + c, p1 = p0 + 4;            // token pairs of this k-step
      // reference values
      {
        float2 vm[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) vm[k] = ld_meta(sb + a.off_vm + (tt[k] * NG + gv) * 4);
        uint32_t bR[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int n = nt * 8 + r;
          float w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float pa = Pa[tt[k] * PR + n];     // 0 for tokens past the context
            w[k] = pa * vm[k].x;
            offR[nt] += pa * vm[k].y;
          }
          split_half2(w[0], w[1], bR[nt][0], bR[nt][2]);
          split_half2(w[2], w[3], bR[nt][1], bR[nt][3]);
        }
        const uint32_t W0 = lds32(sb + a.off_vc + p0 * D + ((8 * gv + r) ^ v_unit_swizzle(p0, D / 4)) * 4);
        const uint32_t W1 = lds32(sb + a.off_vc + p1 * D + ((8 * gv + r) ^ v_unit_swizzle(p1, D / 4)) * 4);
#pragma unroll
        for (int m = 0; m < MTW; ++m) {
          const int mtg = (D == 128) ? m : (warp & 1);
          uint32_t a0, a1, a2, a3;
          a_pairs_4bit<true>(W0, mtg, a0, a1);
          a_pairs_4bit<true>(W1, mtg, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_f16(accR[m][nt], a0, a1, a2, a3, bR[nt][0], bR[nt][1]);
            mma_f16(accR[m][nt], a0, a1, a2, a3, bR[nt][2], bR[nt][3]);
          }
        }
      }
      // residual values: one set of weights per column (its own loop's step)
      if (nr > 0) {
        uint4 bE[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int n = nt * 8 + r;
          const int ri = riB[nt];
          float w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 mm = ld_meta(sb + vrmB[nt] + (tt[k] * NG + gv) * 4);
            const float ps = ri >= 0 ? Ps[tt[k] * PR + n] : 0.f;
            w[k] = ps * mm.x;
            offE[nt] += ps * mm.y;
          }
          split_half2(w[0], w[1], bE[nt].x, bE[nt].z);
          split_half2(w[2], w[3], bE[nt].y, bE[nt].w);
        }
#pragma unroll
        for (int ri = 0; ri < kMaxResPerBlock; ++ri) {
          if (ri >= nr) break;
          const int nt_ri = ((blk.r0 + ri - blk.lb) * blk.gw) >> 3;
          if (a.rbits[ri] == 2) {
            const int sh = 8 * (r & 1);
            const int u = 4 * gv + (r >> 1);
            const uint32_t W0 =
                lds32(sb + a.off_vrc[ri] + p0 * (2 * RB2) + (u ^ v_unit_swizzle(p0, D / 8)) * 4) >> sh;
            const uint32_t W1 =
                lds32(sb + a.off_vrc[ri] + p1 * (2 * RB2) + (u ^ v_unit_swizzle(p1, D / 8)) * 4) >> sh;
#pragma unroll
            for (int m = 0; m < MTW; ++m) {
              const int mtg = (D == 128) ? m : (warp & 1);
              uint32_t a0, a1, a2, a3;
              a_pairs_2bit<true>(W0, mtg, a0, a1);
              a_pairs_2bit<true>(W1, mtg, a2, a3);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt != nt_ri) continue;
                const uint4 bb = sel4(riB[nt] == ri, bE[nt]);
                mma_f16(accE2[m][nt], a0, a1, a2, a3, bb.x, bb.y);
                mma_f16(accE2[m][nt], a0, a1, a2, a3, bb.z, bb.w);
              }
            }
          } else if (RES4) {
            const uint32_t W0 =
                lds32(sb + a.off_vrc[ri] + p0 * D + ((8 * gv + r) ^ v_unit_swizzle(p0, D / 4)) * 4);
            const uint32_t W1 =
                lds32(sb + a.off_vrc[ri] + p1 * D + ((8 * gv + r) ^ v_unit_swizzle(p1, D / 4)) * 4);
#pragma unroll
            for (int m = 0; m < MTW; ++m) {
              const int mtg = (D == 128) ? m : (warp & 1);
              uint32_t a0, a1, a2, a3;
              a_pairs_4bit<true>(W0, mtg, a0, a1);
              a_pairs_4bit<true>(W1, mtg, a2, a3);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt != nt_ri) continue;
                const uint4 bb = sel4(riB[nt] == ri, bE[nt]);
                mma_f16(accE4[RES4 ? m : 0][nt], a0, a1, a2, a3, bb.x, bb.y);
                mma_f16(accE4[RES4 ? m : 0][nt], a0, a1, a2, a3, bb.z, bb.w);
              }
            }
          }
        }
      }
    }
  }

  if (__syncthreads_or(failed)) {
    // a copy never completed: flag it, wait (bounded) for the copies still in flight, leave
    if (threadIdx.x == 0) {
      atomicOr(a.err, 1u);
      for (int t = fail_tile; t < next_issue; ++t)
        mbar_wait_bounded(smem_u32(&bars[t % S]), uint32_t((t / S) & 1), kWaitLimitNs);
    }
    __syncthreads();
    return;
  }

  // ------------------------------------------------------------------ split partials
  // softmax sums: over the 8 row lanes, then over the warps
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = lpart[nt][e];
      v += __shfl_xor_sync(RQ_FULL_MASK, v, 4);
      v += __shfl_xor_sync(RQ_FULL_MASK, v, 8);
      v += __shfl_xor_sync(RQ_FULL_MASK, v, 16);
      if (r == 0) red[warp * NQP + nt * 8 + 2 * c + e] = v;
    }
  // value offsets: over the 4 token lanes of each column
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    offR[nt] += __shfl_xor_sync(RQ_FULL_MASK, offR[nt], 1);
    offR[nt] += __shfl_xor_sync(RQ_FULL_MASK, offR[nt], 2);
    offE[nt] += __shfl_xor_sync(RQ_FULL_MASK, offE[nt], 1);
    offE[nt] += __shfl_xor_sync(RQ_FULL_MASK, offE[nt], 2);
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
  if (threadIdx.x < NQP) {
    float* o = rec_ptr(threadIdx.x);
    if (o) {
      float ls = 0.f;
#pragma unroll
      for (int w = 0; w < kW; ++w) ls += red[w * NQP + threadIdx.x];
      o[0] = mrun[threadIdx.x];
      o[1] = ls;
    }
  }
  // channels of this thread: 32 gv + 4 r + 2 mtg + {0, 1}; columns nt*8 + 2c + {0, 1}
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = nt * 8 + 2 * c + e;
      const float oR = __shfl_sync(RQ_FULL_MASK, offR[nt], (2 * c + e) * 4);
      const float oE = __shfl_sync(RQ_FULL_MASK, offE[nt], (2 * c + e) * 4);
      float* o = rec_ptr(col);
      if (!o) continue;
#pragma unroll
      for (int m = 0; m < MTW; ++m) {
        const int mtg = (D == 128) ? m : (warp & 1);
        const int ch = 32 * gv + 4 * r + 2 * mtg;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {      // hh: row r (j even) or row r+8 (j odd)
          const int j = 2 * mtg + hh;
          const float sc4 = (j & 1) ? 0.0625f : 1.f;      // value codes are normal fp16
          const float sc2 = 1.f / float(1 << (2 * j));
          const float vr = accR[m][nt][2 * hh + e] * sc4 + oR;
          float ve = accE2[m][nt][2 * hh + e] * sc2 + oE;
          if (RES4) ve += accE4[RES4 ? m : 0][nt][2 * hh + e] * sc4;
          o[4 + ch + hh] = vr;
          o[4 + D + ch + hh] = ve;
        }
      }
    }
  }
}

using KernelFn = void (*)(MmaArgs);

template <int D>
KernelFn pick_generic(bool res4) {
  return res4 ? rq_mma_kernel<D, 1, true, -1> : rq_mma_kernel<D, 1, false, -1>;
}

// Variants with the residual-loop count fixed at compile time, for the common blocks: one
// loop of a per-loop call (0 or 1 residual), two loops of a 4-query-head GQA block (2) and
// all four loops of a 4-loop model (3).
KernelFn pick(int D, int nt, bool res4, int nr) {
  if (D == 128 && nt == 1 && !res4) {
    if (nr == 0) return rq_mma_kernel<128, 1, false, 0>;
    if (nr == 1) return rq_mma_kernel<128, 1, false, 1>;
    if (nr == 2) return rq_mma_kernel<128, 1, false, 2>;
    if (nr == 3) return rq_mma_kernel<128, 1, false, 3>;
  }
  if (D == 128 && nt == 1 && res4) {
    if (nr == 1) return rq_mma_kernel<128, 1, true, 1>;
    if (nr == 3) return rq_mma_kernel<128, 1, true, 3>;
  }
  if (D == 64 && nt == 1 && !res4) {
    if (nr == 0) return rq_mma_kernel<64, 1, false, 0>;
    if (nr == 1) return rq_mma_kernel<64, 1, false, 1>;
    if (nr == 3) return rq_mma_kernel<64, 1, false, 3>;
  }
  (void)nt;                                     // blocks hold one n-tile (8 columns)
  return D == 128 ? pick_generic<128>(res4) : pick_generic<64>(res4);
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
      for (int nt : {1})
        for (bool r4 : {false, true})
          for (int nr = -1; nr <= kMaxResPerBlock; ++nr) {
            cudaError_t e = cudaFuncSetAttribute(pick(D, nt, r4, nr),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 200 * 1024);
            if (e != cudaSuccess) err[dev] = e;
          }
  });
  return err[dev];
}

// CTAs of a kernel variant resident per SM with `smem` bytes of dynamic shared memory.
int resident_ctas(int D, int nt, bool res4, int nr, size_t smem) {
  int n = 0;
  if (prepare_kernels() == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pick(D, nt, res4, nr), kW * 32, smem) ==
          cudaSuccess &&
      n > 0)
    return n;
  const int by_smem = int((227 * 1024) / (smem + 1024));   // no device: shared-memory bound
  return by_smem < 1 ? 1 : (by_smem > 8 ? 8 : by_smem);
}

struct BlockLaunch {
  MmaArgs a;
  int nt;
  bool res4;
  size_t smem;
};

// Arguments, stage layout and shared memory of one query block (no launch).
bool build_block(const rq_shape& s, const rq_cache& cache, const QueryBlock& bq, BlockLaunch& bl) {
  MmaArgs& a = bl.a;
  memset(&a, 0, sizeof(a));
  const int D = s.head_dim, NG = D / 32;
  a.kc = cache.ref_codes[0];
  a.km = cache.ref_meta[0];
  a.vc = cache.ref_codes[1];
  a.vm = cache.ref_meta[1];
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
    a.krc[ri] = cache.res_codes[0][l];
    a.krm[ri] = cache.res_meta[0][l];
    a.ka[ri] = cache.alpha[0][l];
    a.vrc[ri] = cache.res_codes[1][l];
    a.vrm[ri] = cache.res_meta[1][l];
    a.va[ri] = cache.alpha[1][l];
    a.off_krc[ri] = off; off += kT * D * bits / 8;
    a.off_krm[ri] = off; off += kT * NG * 4;
    a.off_ka[ri] = off;  off += kT * 2;
    a.off_vrc[ri] = off; off += kT * D * bits / 8;
    a.off_vrm[ri] = off; off += kT * NG * 4;
    a.off_va[ri] = off;  off += kT * 2;
  }
  a.stage_bytes = off;
  a.blk = bq;
  const int nq = bq.gw * bq.nl;
  bl.nt = nq <= 8 ? 1 : (nq <= 16 ? 2 : 4);
  bl.res4 = res4;
  // most resident CTAs per SM first (latency hiding), then the deepest pipeline
  int best_ctas = 0;
  for (int stages = 3; stages >= 2; --stages) {
    const size_t sm = smem_layout(D, bl.nt, res4, stages, a.stage_bytes).total;
    if (sm > 200 * 1024) continue;
    const int ctas = resident_ctas(D, bl.nt, res4, bq.nr, sm);
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
constexpr int kMaxBlockColumns = 8;

int plan_query_blocks(int g, int loop_begin, int loop_count, int L, QueryBlock* out, int max_out) {
  int gw = 1;
  while (gw < g && gw < 8) gw <<= 1;
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
        if (res && nres == kMaxResPerBlock) break;
        nres += res;
        ++nl;
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

SplitPlan plan_splits_rq(const rq_shape& s, int loop_begin, int loop_count, int max_ctx) {
  // the resident CTAs per SM follow the largest shared-memory block of the call
  QueryBlock blocks[64];
  const int g = s.n_q_heads / s.n_kv_heads;
  const int nb = plan_query_blocks(g, loop_begin, loop_count, s.n_loops, blocks, 64);
  rq_cache dummy;
  memset(&dummy, 0, sizeof(dummy));
  int ctas = 0;
  for (int i = 0; i < nb; ++i) {
    BlockLaunch bl;
    if (!build_block(s, dummy, blocks[i], bl)) continue;
    const int n = resident_ctas(s.head_dim, bl.nt, bl.res4, blocks[i].nr, bl.smem);
    if (ctas == 0 || n < ctas) ctas = n;
  }
  return plan_splits_for(s, max_ctx, ctas > 0 ? ctas : 1, kT);
}

cudaError_t launch_rq_decode_mma(const rq_shape& s, const rq_cache& cache, const uint16_t* q,
                                 int loop_begin, int loop_count, const int32_t* ctx_lens,
                                 int n_splits, int tokens_per_split, float* part, unsigned* err,
                                 cudaStream_t stream) {
  cudaError_t e = prepare_kernels();
  if (e != cudaSuccess) return e;
  QueryBlock blocks[64];
  const int g = s.n_q_heads / s.n_kv_heads;
  const int nb = plan_query_blocks(g, loop_begin, loop_count, s.n_loops, blocks, 64);
  if (nb < 0) return cudaErrorInvalidConfiguration;
  const float scale = s.softmax_scale > 0.f ? s.softmax_scale : 1.0f / sqrtf(float(s.head_dim));
  for (int bi = 0; bi < nb; ++bi) {
    BlockLaunch bl;
    if (!build_block(s, cache, blocks[bi], bl)) return cudaErrorInvalidConfiguration;
    MmaArgs& a = bl.a;
    a.ksigns = cache.rot_signs[0];
    a.q = q;
    a.ctx_lens = ctx_lens;
    a.part = part;
    a.err = err;
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
    dim3 grid(n_splits, s.n_kv_heads, s.batch);
    pick(s.head_dim, bl.nt, bl.res4, blocks[bi].nr)<<<grid, kW * 32, bl.smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace rq
