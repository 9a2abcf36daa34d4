// ResidualQuant split-KV decode attention on the tensor cores (sm_103a).
//
// Per CTA: one (split of the context, kv-head, sequence); 4 warps; 64-token tiles of every
// packed array are staged in shared memory by 1-D bulk (TMA) copies through a multi-stage
// mbarrier pipeline.  For a loop-l query q and token t (rit.work summary, "How each pass's
// KV cache is reconstructed": reference and residuals rebuilt inside attention)
//   score_t = a_t * sum_g s^r_g,t (q_g . c^r_g,t) + z^r_g,t sum(q_g)
//           +       sum_g s^e_g,t (q'_g . c^e_g,t) + z^e_g,t sum(q'_g),     q' = R q
//   acc_ref += p_t a_t (s^r c^r + z^r),  acc_res += p_t (s^e c^e + z^e)   (rotated domain)
// The code dot products and the P.V products run as mma.sync m16n8k16 (f16 in, f32 acc):
//   scores: M = 16 tokens, N = 8 queries, K = 16 channels of one 32-channel group;
//   values: M = 16 channels of one group, N = 8 queries, K = 16 tokens.
// A pair of packed codes becomes an f16x2 operand with one LOP3 and one packed subtract:
// the code bits, masked in place, sit in the low mantissa bits of 1024 (0x6400), and
// subtracting 1024 leaves the code times a power of two fixed by its bit position; that
// power is folded into the query fragments (scores) or removed per output row at the end
// (values).  Products of fp16 operands are exact in the fp32 accumulators.  The other
// operand (queries, softmax weights) is split into an fp16 high part and an fp16 low part
// (two MMAs), so it carries about 22 significant bits.
// Per-(token, group) steps and offsets are applied in fp32 to the score fragments and
// folded into P for the values; the offsets' value terms are accumulated separately.
#include <mutex>

#include "rq_common.cuh"
#include "rq_kernels.h"
#include "rq_ptx.cuh"

namespace rq {
namespace {

constexpr int kT = 64;                        // tokens per tile
constexpr int kW = 4;                         // warps per CTA
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kCodeUnit = 1.0f;    // fp16 code operands hold the code values exactly

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

__device__ __forceinline__ float2 ld_meta(const uint8_t* p) {  // (step, offset) fp16 pair
  const __half2 h = *reinterpret_cast<const __half2*>(p);
  return __half22float2(h);
}

__device__ __forceinline__ float ld_half(const uint8_t* p) {
  return __half2float(*reinterpret_cast<const __half*>(p));
}

template <int D, int NT, bool RES4>
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
  const int nr = blk.nr;

  const SmemLayout lay = smem_layout(D, NT, nr, a.n_stages, a.stage_bytes);
  uint4* QF = reinterpret_cast<uint4*>(smem + lay.qf);    // {b0, b1} high parts, {b0, b1} low
  uint4* QRF = reinterpret_cast<uint4*>(smem + lay.qrf);
  float* Qsum = reinterpret_cast<float*>(smem + lay.qsum);
  float* QRS = reinterpret_cast<float*>(smem + lay.qrs);
  float* Ps = reinterpret_cast<float*>(smem + lay.ps);
  float* Pa = reinterpret_cast<float*>(smem + lay.pa);
  float* red = reinterpret_cast<float*>(smem + lay.red);
  float* mrun = reinterpret_cast<float*>(smem + lay.mrun);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);

  // ------------------------------------------------------------------ query preparation
  {
    uint32_t* z32 = reinterpret_cast<uint32_t*>(smem + lay.qf);
    const int nz = (lay.mrun - lay.qf) / 4;     // QF, QRF, Qsum, QRS, Ps, Pa, red
    for (int i = threadIdx.x; i < nz; i += blockDim.x) z32[i] = 0u;
    for (int i = threadIdx.x; i < NQP; i += blockDim.x) mrun[i] = -INFINITY;
  }
  __syncthreads();
  for (int n = warp; n < NQP; n += kW) {
    const int li = n / blk.gw;
    const int gi = blk.gi0 + n % blk.gw;
    const bool real = li < blk.nl && gi < a.g;
    const int l = blk.lb + li;
    float v[P], rr[P];
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
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      rr[j] *= inv_sqrt_d;
      s1 += v[j];
      s2 += rr[j];
    }
#pragma unroll
    for (int o = 1; o < 32 / P; o <<= 1) {
      s1 += __shfl_xor_sync(RQ_FULL_MASK, s1, o);
      s2 += __shfl_xor_sync(RQ_FULL_MASK, s2, o);
    }
    const int ri = (real && l != a.L - 1) ? l - blk.r0 : -1;
    const int grp = (lane * P) >> 5;
    if ((lane & (32 / P - 1)) == 0) {
      Qsum[grp * NQP + n] = s1;
      if (ri >= 0) QRS[(ri * NG + grp) * 8 + (n & 7)] = s2;
    }
    const int nt = n >> 3, nn = n & 7;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const int ch = lane * P + j, gq = ch >> 5, cl = ch & 31;
      {  // 4-bit mapping: slot (c4, s, hi, e) <- channel 8 c4 + 2 s + hi + 4 e, scale 16^-hi
        const int c4 = cl >> 3, w8 = cl & 7, s = (w8 >> 1) & 1, hi = w8 & 1, e = w8 >> 2;
        __half* dst = reinterpret_cast<__half*>(&QF[((gq * 2 + s) * NT + nt) * 32 + nn * 4 + c4]);
        split_half(hi ? v[j] * 0.0625f : v[j], dst[hi * 2 + e], dst[4 + hi * 2 + e]);
      }
      if (ri >= 0) {
        __half* base = reinterpret_cast<__half*>(QRF);
        if (a.rbits[ri] == 4) {
          const int c4 = cl >> 3, w8 = cl & 7, s = (w8 >> 1) & 1, hi = w8 & 1, e = w8 >> 2;
          __half* dst = base + (((ri * NG + gq) * 2 + s) * 32 + nn * 4 + c4) * 8;
          split_half(hi ? rr[j] * 0.0625f : rr[j], dst[hi * 2 + e], dst[4 + hi * 2 + e]);
        } else {  // 2-bit mapping: slot (cq, s, hi, e) <- channel 16(cq/2) + 4(cq%2) + 2s + hi + 8e
          const int e = (cl >> 3) & 1, cq = 2 * (cl >> 4) + ((cl & 7) >> 2), jj = cl & 3;
          const int s = jj >> 1, hi = jj & 1;
          const float sc = (jj == 0) ? 1.f : (jj == 1) ? 0.25f : (jj == 2) ? 0.0625f : 0.015625f;
          __half* dst = base + (((ri * NG + gq) * 2 + s) * 32 + nn * 4 + cq) * 8;
          split_half(rr[j] * sc, dst[hi * 2 + e], dst[4 + hi * 2 + e]);
        }
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
    for (int ri = 0; ri < nr; ++ri) {
      const int rb = D * a.rbits[ri] / 8;
      bulk_g2s(dst + a.off_krc[ri], a.krc[ri] + tok * rb, kT * rb, bar);
      bulk_g2s(dst + a.off_krm[ri], a.krm[ri] + tok * NG * 2, kT * NG * 4, bar);
      bulk_g2s(dst + a.off_ka[ri], a.ka[ri] + tok, kT * 2, bar);
      bulk_g2s(dst + a.off_vrc[ri], a.vrc[ri] + tok * rb, kT * rb, bar);
      bulk_g2s(dst + a.off_vrm[ri], a.vrm[ri] + tok * NG * 2, kT * NG * 4, bar);
      bulk_g2s(dst + a.off_va[ri], a.va[ri] + tok, kT * 2, bar);
    }
  };
  int next_issue = 0;   // tiles issued so far (thread 0)
  if (threadIdx.x == 0) {
    for (; next_issue < S && next_issue < ntiles; ++next_issue) issue(next_issue);
  }

  // per-column facts for this thread's score columns (nt*8 + 2c + e)
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
    float sc[NT][4];
    {
      float Sref[NT][4], Sres[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) Sref[nt][k] = Sres[nt][k] = 0.f;
#pragma unroll
      for (int gq = 0; gq < NG; ++gq) {
        const uint32_t wl = lds32(sb + a.off_kc + tr0 * RB4 + 16 * gq + 4 * c);
        const uint32_t wh = lds32(sb + a.off_kc + tr1 * RB4 + 16 * gq + 4 * c);
        const float2 m0 = ld_meta(sb + a.off_km + (tr0 * NG + gq) * 4);
        const float2 m1 = ld_meta(sb + a.off_km + (tr1 * NG + gq) * 4);
        float Dg[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int k = 0; k < 4; ++k) Dg[nt][k] = 0.f;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const uint32_t xl = s ? (wl >> 8) : wl, xh = s ? (wh >> 8) : wh;
          const uint32_t a0 = code_pair(xl, 0x000F000Fu), a1 = code_pair(xh, 0x000F000Fu);
          const uint32_t a2 = code_pair(xl, 0x00F000F0u), a3 = code_pair(xh, 0x00F000F0u);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 bq = QF[((gq * 2 + s) * NT + nt) * 32 + lane];
            mma_f16(Dg[nt], a0, a1, a2, a3, bq.x, bq.y);
            mma_f16(Dg[nt], a0, a1, a2, a3, bq.z, bq.w);
          }
        }
        const float s0 = m0.x * kCodeUnit, s1 = m1.x * kCodeUnit;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float2 qs = *reinterpret_cast<const float2*>(&Qsum[gq * NQP + nt * 8 + 2 * c]);
          Sref[nt][0] += s0 * Dg[nt][0] + m0.y * qs.x;
          Sref[nt][1] += s0 * Dg[nt][1] + m0.y * qs.y;
          Sref[nt][2] += s1 * Dg[nt][2] + m1.y * qs.x;
          Sref[nt][3] += s1 * Dg[nt][3] + m1.y * qs.y;
        }
      }
      for (int ri = 0; ri < nr; ++ri) {
        const int l = blk.r0 + ri;
        const int nt_ri = ((l - blk.lb) * blk.gw) >> 3;
        const bool two = a.rbits[ri] == 2;
#pragma unroll
        for (int gq = 0; gq < NG; ++gq) {
          uint32_t wl, wh;
          if (two) {
            const int off = a.off_krc[ri] + 8 * gq + 4 * (c >> 1);
            wl = lds32(sb + off + tr0 * RB2) >> (8 * (c & 1));
            wh = lds32(sb + off + tr1 * RB2) >> (8 * (c & 1));
          } else {
            wl = lds32(sb + a.off_krc[ri] + tr0 * RB4 + 16 * gq + 4 * c);
            wh = lds32(sb + a.off_krc[ri] + tr1 * RB4 + 16 * gq + 4 * c);
          }
          const float2 m0 = ld_meta(sb + a.off_krm[ri] + (tr0 * NG + gq) * 4);
          const float2 m1 = ld_meta(sb + a.off_krm[ri] + (tr1 * NG + gq) * 4);
          float Dg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            uint32_t a0, a1, a2, a3;
            if (two) {
              const uint32_t mlo = 0x00030003u << (4 * s), mhi = 0x00030003u << (4 * s + 2);
              a0 = code_pair(wl, mlo);
              a1 = code_pair(wh, mlo);
              a2 = code_pair(wl, mhi);
              a3 = code_pair(wh, mhi);
            } else {
              const uint32_t xl = s ? (wl >> 8) : wl, xh = s ? (wh >> 8) : wh;
              a0 = code_pair(xl, 0x000F000Fu);
              a1 = code_pair(xh, 0x000F000Fu);
              a2 = code_pair(xl, 0x00F000F0u);
              a3 = code_pair(xh, 0x00F000F0u);
            }
            const uint4 bq = QRF[((ri * NG + gq) * 2 + s) * 32 + lane];
            mma_f16(Dg, a0, a1, a2, a3, bq.x, bq.y);
            mma_f16(Dg, a0, a1, a2, a3, bq.z, bq.w);
          }
          const float2 qs = *reinterpret_cast<const float2*>(&QRS[(ri * NG + gq) * 8 + 2 * c]);
          const float s0 = m0.x * kCodeUnit, s1 = m1.x * kCodeUnit;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (nt != nt_ri) continue;
            Sres[nt][0] += s0 * Dg[0] + m0.y * qs.x;
            Sres[nt][1] += s0 * Dg[1] + m0.y * qs.y;
            Sres[nt][2] += s1 * Dg[2] + m1.y * qs.x;
            Sres[nt][3] += s1 * Dg[3] + m1.y * qs.y;
          }
        }
      }
      // combine: score = a_t * ref part + residual part (final loop: the reference alone)
      const bool v0 = t0 + tr0 < t_end, v1 = t0 + tr1 < t_end;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = nt * 8 + 2 * c + e;
          const int li = col / blk.gw;
          const int l = blk.lb + li;
          float s_0 = Sref[nt][e], s_1 = Sref[nt][2 + e];
          if (li < blk.nl && l != a.L - 1) {
            const int ri = l - blk.r0;
            s_0 = ld_half(sb + a.off_ka[ri] + tr0 * 2) * s_0 + Sres[nt][e];
            s_1 = ld_half(sb + a.off_ka[ri] + tr1 * 2) * s_1 + Sres[nt][2 + e];
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
    const bool v0 = t0 + tr0 < t_end, v1 = t0 + tr1 < t_end;
    // rescale of the value-offset sums, kept per B-fragment column nt*8 + r
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
        const int li = col / blk.gw;
        const int l = blk.lb + li;
        float a0v = 1.f, a1v = 1.f;
        if (li < blk.nl && l != a.L - 1) {
          const int ri = l - blk.r0;
          a0v = ld_half(sb + a.off_va[ri] + tr0 * 2);
          a1v = ld_half(sb + a.off_va[ri] + tr1 * 2);
        }
        Ps[tr0 * NQP + col] = p0;
        Ps[tr1 * NQP + col] = p1;
        Pa[tr0 * NQP + col] = v0 ? p0 * a0v : 0.f;
        Pa[tr1 * NQP + col] = v1 ? p1 * a1v : 0.f;
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
      const int tt[4] = {16 * ks + 2 * c, 16 * ks + 2 * c + 1, 16 * ks + 2 * c + 8,
                         16 * ks + 2 * c + 9};
      bool val[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) val[k] = t0 + tt[k] < t_end;
      const int p0 = 8 * ks + c, p1 = p0 + 4;            // token pairs of this k-step
      // reference values
      {
        float vs[4], vz[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 mm = ld_meta(sb + a.off_vm + (tt[k] * NG + gv) * 4);
          vs[k] = mm.x;
          vz[k] = mm.y;
        }
        uint32_t bR[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int n = nt * 8 + r;
          float w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float pa = Pa[tt[k] * NQP + n];
            w[k] = val[k] ? pa * vs[k] : 0.f;
            offR[nt] += val[k] ? pa * vz[k] : 0.f;
          }
          split_half2(w[0], w[1], bR[nt][0], bR[nt][2]);
          split_half2(w[2], w[3], bR[nt][1], bR[nt][3]);
        }
        const uint32_t W0 = lds32(sb + a.off_vc + p0 * D + (8 * gv + r) * 4);
        const uint32_t W1 = lds32(sb + a.off_vc + p1 * D + (8 * gv + r) * 4);
#pragma unroll
        for (int m = 0; m < MTW; ++m) {
          const int mtg = (D == 128) ? m : (warp & 1);
          const uint32_t x0 = mtg ? (W0 >> 8) : W0, x1 = mtg ? (W1 >> 8) : W1;
          const uint32_t a0 = code_pair(x0, 0x000F000Fu), a1 = code_pair(x0, 0x00F000F0u);
          const uint32_t a2 = code_pair(x1, 0x000F000Fu), a3 = code_pair(x1, 0x00F000F0u);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_f16(accR[m][nt], a0, a1, a2, a3, bR[nt][0], bR[nt][1]);
            mma_f16(accR[m][nt], a0, a1, a2, a3, bR[nt][2], bR[nt][3]);
          }
        }
      }
      // residual values of each loop in the block
      for (int ri = 0; ri < nr; ++ri) {
        const int l = blk.r0 + ri;
        const int nt_ri = ((l - blk.lb) * blk.gw) >> 3;
        const int n = nt_ri * 8 + r;
        const int li = n / blk.gw;
        const bool mine = li < blk.nl && blk.lb + li == l;
        float w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 mm = ld_meta(sb + a.off_vrm[ri] + (tt[k] * NG + gv) * 4);
          const float ps = Ps[tt[k] * NQP + n];
          const bool use = mine && val[k];
          w[k] = use ? ps * mm.x : 0.f;
          const float oz = use ? ps * mm.y : 0.f;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            if (nt == nt_ri) offE[nt] += oz;
        }
        uint32_t b0, b1, b0l, b1l;
        split_half2(w[0], w[1], b0, b0l);
        split_half2(w[2], w[3], b1, b1l);
        if (a.rbits[ri] == 2) {
          const int sh = 8 * (r & 1);
          const uint32_t W0 = lds32(sb + a.off_vrc[ri] + p0 * (2 * RB2) + (4 * gv + (r >> 1)) * 4) >> sh;
          const uint32_t W1 = lds32(sb + a.off_vrc[ri] + p1 * (2 * RB2) + (4 * gv + (r >> 1)) * 4) >> sh;
#pragma unroll
          for (int m = 0; m < MTW; ++m) {
            const int mtg = (D == 128) ? m : (warp & 1);
            const uint32_t mlo = 0x00030003u << (4 * mtg), mhi = 0x00030003u << (4 * mtg + 2);
            const uint32_t a0 = code_pair(W0, mlo), a1 = code_pair(W0, mhi);
            const uint32_t a2 = code_pair(W1, mlo), a3 = code_pair(W1, mhi);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              if (nt == nt_ri) {
                mma_f16(accE2[m][nt], a0, a1, a2, a3, b0, b1);
                mma_f16(accE2[m][nt], a0, a1, a2, a3, b0l, b1l);
              }
          }
        } else if (RES4) {
          const uint32_t W0 = lds32(sb + a.off_vrc[ri] + p0 * D + (8 * gv + r) * 4);
          const uint32_t W1 = lds32(sb + a.off_vrc[ri] + p1 * D + (8 * gv + r) * 4);
#pragma unroll
          for (int m = 0; m < MTW; ++m) {
            const int mtg = (D == 128) ? m : (warp & 1);
            const uint32_t x0 = mtg ? (W0 >> 8) : W0, x1 = mtg ? (W1 >> 8) : W1;
            const uint32_t a0 = code_pair(x0, 0x000F000Fu), a1 = code_pair(x0, 0x00F000F0u);
            const uint32_t a2 = code_pair(x1, 0x000F000Fu), a3 = code_pair(x1, 0x00F000F0u);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              if (nt == nt_ri) {
                mma_f16(accE4[RES4 ? m : 0][nt], a0, a1, a2, a3, b0, b1);
                mma_f16(accE4[RES4 ? m : 0][nt], a0, a1, a2, a3, b0l, b1l);
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
          const float sc4 = (j & 1) ? kCodeUnit / 16.f : kCodeUnit;
          const float sc2 = kCodeUnit / float(1 << (2 * j));
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

template <int D, int NT, bool RES4>
cudaError_t launch_variant(const MmaArgs& a, dim3 grid, size_t smem, cudaStream_t stream) {
  auto k = rq_mma_kernel<D, NT, RES4>;
  // opt in to the largest dynamic shared memory once per kernel variant and device
  static std::once_flag once[64];
  static cudaError_t set_err[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    set_err[dev] = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  });
  if (set_err[dev] != cudaSuccess) return set_err[dev];
  k<<<grid, kW * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const MmaArgs& a, int nt, bool res4, dim3 grid, size_t smem,
                     cudaStream_t stream) {
  if (nt == 1) return res4 ? launch_variant<D, 1, true>(a, grid, smem, stream)
                           : launch_variant<D, 1, false>(a, grid, smem, stream);
  if (nt == 2) return res4 ? launch_variant<D, 2, true>(a, grid, smem, stream)
                           : launch_variant<D, 2, false>(a, grid, smem, stream);
  return res4 ? launch_variant<D, 4, true>(a, grid, smem, stream)
              : launch_variant<D, 4, false>(a, grid, smem, stream);
}

}  // namespace

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
      while (l + nl < lend && (nl + 1) * gw <= 32) {
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

size_t stage_bytes_for(int D, const int8_t* res_bits, const QueryBlock& bq) {
  const int NG = D / 32;
  size_t s = 2 * (size_t(kT) * D / 2 + size_t(kT) * NG * 4);
  for (int ri = 0; ri < bq.nr; ++ri)
    s += 2 * (size_t(kT) * D * res_bits[bq.r0 + ri] / 8 + size_t(kT) * NG * 4 + kT * 2);
  return s;
}

cudaError_t launch_rq_decode_mma(const rq_shape& s, const rq_cache& cache, const uint16_t* q,
                                 int loop_begin, int loop_count, const int32_t* ctx_lens,
                                 int n_splits, int tokens_per_split, float* part, unsigned* err,
                                 cudaStream_t stream) {
  QueryBlock blocks[64];
  const int g = s.n_q_heads / s.n_kv_heads;
  const int nb = plan_query_blocks(g, loop_begin, loop_count, s.n_loops, blocks, 64);
  if (nb < 0) return cudaErrorInvalidConfiguration;
  const int D = s.head_dim, NG = D / 32;
  const float scale = s.softmax_scale > 0.f ? s.softmax_scale : 1.0f / sqrtf(float(D));
  for (int bi = 0; bi < nb; ++bi) {
    const QueryBlock& bq = blocks[bi];
    MmaArgs a;
    memset(&a, 0, sizeof(a));
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
      a.off_ka[ri] = off; off += kT * 2;
      a.off_vrc[ri] = off; off += kT * D * bits / 8;
      a.off_vrm[ri] = off; off += kT * NG * 4;
      a.off_va[ri] = off; off += kT * 2;
    }
    a.stage_bytes = off;
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
    a.blk = bq;
    a.scale_log2 = scale * kLog2e;
    const int nq = bq.gw * bq.nl;
    const int nt = nq <= 8 ? 1 : (nq <= 16 ? 2 : 4);
    int stages = 3;
    size_t smem = 0;
    for (; stages >= 1; --stages) {
      smem = smem_layout(D, nt, bq.nr, stages, a.stage_bytes).total;
      if (smem <= 200 * 1024) break;
    }
    if (stages < 1) return cudaErrorInvalidConfiguration;
    a.n_stages = stages;
    dim3 grid(n_splits, s.n_kv_heads, s.batch);
    cudaError_t e = (D == 128) ? launch_d<128>(a, nt, res4, grid, smem, stream)
                               : launch_d<64>(a, nt, res4, grid, smem, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace rq
