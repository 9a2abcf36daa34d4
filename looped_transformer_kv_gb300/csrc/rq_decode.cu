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

constexpr int kWarps = 4;
constexpr int kChunk = 32;                   // tokens per warp iteration (one per lane)
constexpr int kCtaTokens = kWarps * kChunk;  // tokens per CTA iteration

struct DecodeArgs {
  rq_cache cache;
  const uint16_t* q;
  const int32_t* ctx_lens;
  float* ws;
  int B, Hq, H, L, cap, g, loop_begin, loop_count, n_splits, tokens_per_split;
  int q0, nq;  // query block [q0, q0 + nq) of the g * loop_count queries of a kv-head
  float scale_log2;
  int8_t res_bits[RQ_MAX_LOOPS];
};

// Unpack 32 4-bit codes (16 bytes) or 32 2-bit codes (8 bytes) to floats.
__device__ __forceinline__ void unpack32_4(const uint4 r, float (&c)[32]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int k = 0; k < 32; ++k) c[k] = float((w[k >> 3] >> (4 * (k & 7))) & 0xFu);
}
__device__ __forceinline__ void unpack32_2(const uint2 r, float (&c)[32]) {
  const uint32_t w[2] = {r.x, r.y};
#pragma unroll
  for (int k = 0; k < 32; ++k) c[k] = float((w[k >> 4] >> (2 * (k & 15))) & 0x3u);
}

__device__ __forceinline__ float dot32(const float (&c)[32], const float* qs) {
  const float4* q4 = reinterpret_cast<const float4*>(qs);
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float4 v = q4[k];
    acc = fmaf(c[4 * k], v.x, acc);
    acc = fmaf(c[4 * k + 1], v.y, acc);
    acc = fmaf(c[4 * k + 2], v.z, acc);
    acc = fmaf(c[4 * k + 3], v.w, acc);
  }
  return acc;
}

__device__ __forceinline__ void half2_bits(uint32_t w, float& s, float& z) {
  s = half_bits_to_float(uint16_t(w & 0xFFFFu));
  z = half_bits_to_float(uint16_t(w >> 16));
}

// Codes of this lane's P channels in a V row stored in token pairs.
template <int P>
__device__ __forceinline__ uint32_t load_v_lane_codes(const uint8_t* slot, int64_t t, int bits,
                                                      int lane) {
  const int row = P * 32 * bits / 8;
  const int lane_bits = P * bits;
  const int bit0 = lane * lane_bits;
  const int k = bit0 >> 3;
  if (lane_bits == 16) {
    return *reinterpret_cast<const uint16_t*>(slot + vpair_offset(t, k, row));
  }
  uint32_t byte = slot[vpair_offset(t, k, row)];
  return lane_bits == 8 ? byte : ((byte >> (bit0 & 7)) & 0xFu);
}

template <int D, int NQ>
__global__ void __launch_bounds__(kWarps * 32) rq_split_kernel(DecodeArgs a) {
  constexpr int P = D / 32;
  constexpr int NG = D / kGroup;
  __shared__ __align__(16) float q_sm[NQ][D];    // scaled queries
  __shared__ __align__(16) float qr_sm[NQ][D];   // scaled rotated queries R q
  __shared__ float qs_sm[NQ][NG], qrs_sm[NQ][NG];
  __shared__ float p_sm[kWarps][kChunk][NQ];
  __shared__ float m_sm[kWarps][NQ], l_sm[kWarps][NQ];
  __shared__ __align__(16) float acc_sm[kWarps][NQ][2][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int L = a.L;
  const int ctx = min(a.ctx_lens[b], a.cap);
  const int t_begin = split * a.tokens_per_split;
  const int t_end = min(ctx, t_begin + a.tokens_per_split);

  // query n of this block: global index qn = q0 + n -> loop li = qn / g, head gi = qn % g
  int lq[NQ];
#pragma unroll
  for (int n = 0; n < NQ; ++n) {
    const int qn = a.q0 + min(n, a.nq - 1);
    lq[n] = a.loop_begin + qn / a.g;
  }

  // ---- query prep: scale, rotate (R q = H (signs * q) / sqrt(d)), group sums ----
  for (int n = warp; n < NQ; n += kWarps) {
    const int qn = a.q0 + min(n, a.nq - 1);
    const int li = qn / a.g, gi = qn % a.g;
    const int hq = h * a.g + gi;
    const uint16_t* qp = a.q + ((int64_t(b) * a.Hq + hq) * a.loop_count + li) * D + lane * P;
    const int8_t* sg = a.cache.rot_signs[0] + int64_t(h) * D + lane * P;
    float v[P], r[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
      v[j] = bf16_bits_to_float(qp[j]) * a.scale_log2;
      r[j] = v[j] * float(sg[j]);
    }
    warp_fwht<P>(r, lane);
    const float inv_sqrt_d = (D == 128) ? 0.08838834764831845f : 0.125f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      r[j] *= inv_sqrt_d;
      q_sm[n][lane * P + j] = v[j];
      qr_sm[n][lane * P + j] = r[j];
    }
    // group sums: group of channel lane*P is lane*P/32; LPG = 32/P lanes per group
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      s1 += v[j];
      s2 += r[j];
    }
#pragma unroll
    for (int o = 1; o < 32 / P; o <<= 1) {
      s1 += __shfl_xor_sync(RQ_FULL_MASK, s1, o);
      s2 += __shfl_xor_sync(RQ_FULL_MASK, s2, o);
    }
    if (lane % (32 / P) == 0) {
      qs_sm[n][lane * P / 32] = s1;
      qrs_sm[n][lane * P / 32] = s2;
    }
  }
  __syncthreads();

  const int64_t slot = int64_t(b) * a.H + h;
  const uint8_t* kref = a.cache.ref_codes[0] + slot * a.cap * (D / 2);
  const uint16_t* kref_meta = a.cache.ref_meta[0] + slot * a.cap * (2 * NG);
  const uint8_t* vref = a.cache.ref_codes[1] + slot * a.cap * (D / 2);
  const uint16_t* vref_meta = a.cache.ref_meta[1] + slot * a.cap * (2 * NG);

  const int l_first = lq[0], l_last = lq[NQ - 1];

  float m_run[NQ], l_lane[NQ], acc_ref[NQ][P], acc_res[NQ][P];
#pragma unroll
  for (int n = 0; n < NQ; ++n) {
    m_run[n] = -INFINITY;
    l_lane[n] = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) acc_ref[n][j] = acc_res[n][j] = 0.f;
  }

  for (int c0 = t_begin + warp * kChunk; c0 < t_end; c0 += kCtaTokens) {
    const int t = c0 + lane;
    const bool valid = t < t_end;
    const int tl = valid ? t : c0;  // clamp loads of idle lanes to a valid token
    // ---------------- scores (lane = token) ----------------
    float sref[NQ], sres[NQ];
#pragma unroll
    for (int n = 0; n < NQ; ++n) sref[n] = sres[n] = 0.f;
    for (int g = 0; g < NG; ++g) {
      float c[32], s, z;
      unpack32_4(*reinterpret_cast<const uint4*>(kref + int64_t(tl) * (D / 2) + 16 * g), c);
      half2_bits(*reinterpret_cast<const uint32_t*>(kref_meta + int64_t(tl) * 2 * NG + 2 * g), s, z);
#pragma unroll
      for (int n = 0; n < NQ; ++n)
        sref[n] += s * dot32(c, &q_sm[n][32 * g]) + z * qs_sm[n][g];
      for (int l = l_first; l <= l_last; ++l) {
        if (l == L - 1) continue;
        const int bits = a.res_bits[l];
        const int row = D * bits / 8;
        const uint8_t* rc = a.cache.res_codes[0][l] + slot * a.cap * row + int64_t(tl) * row;
        if (bits == 2)
          unpack32_2(*reinterpret_cast<const uint2*>(rc + 8 * g), c);
        else
          unpack32_4(*reinterpret_cast<const uint4*>(rc + 16 * g), c);
        half2_bits(*reinterpret_cast<const uint32_t*>(a.cache.res_meta[0][l] +
                                                      (slot * a.cap + tl) * 2 * NG + 2 * g),
                   s, z);
#pragma unroll
        for (int n = 0; n < NQ; ++n)
          if (lq[n] == l) sres[n] += s * dot32(c, &qr_sm[n][32 * g]) + z * qrs_sm[n][g];
      }
    }
    float score[NQ];
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
      const int l = lq[n];
      float sc = sref[n];
      if (l != L - 1) {
        const float al = half_bits_to_float(a.cache.alpha[0][l][slot * a.cap + tl]);
        sc = al * sref[n] + sres[n];
      }
      score[n] = valid ? sc : -INFINITY;
    }
    // ---------------- online softmax (warp-uniform running max) ----------------
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
      const float mc = warp_max(score[n]);
      const float m_new = fmaxf(m_run[n], mc);
      const float corr = (m_run[n] == -INFINITY) ? 0.f : exp2f(m_run[n] - m_new);
      const float p = valid ? exp2f(score[n] - m_new) : 0.f;
      l_lane[n] = l_lane[n] * corr + p;
#pragma unroll
      for (int j = 0; j < P; ++j) {
        acc_ref[n][j] *= corr;
        acc_res[n][j] *= corr;
      }
      m_run[n] = m_new;
      p_sm[warp][lane][n] = p;
    }
    __syncwarp();
    // ---------------- values (lane = channels lane*P .. lane*P+P-1) ----------------
    const int nvalid = min(kChunk, t_end - c0);
    const int grp = lane * P / 32;
    for (int tt = 0; tt < nvalid; ++tt) {
      const int64_t tv = c0 + tt;
      float s, z;
      half2_bits(*reinterpret_cast<const uint32_t*>(vref_meta + tv * 2 * NG + 2 * grp), s, z);
      const uint32_t cr = load_v_lane_codes<P>(vref, tv, 4, lane);
      float vr[P];
#pragma unroll
      for (int j = 0; j < P; ++j) vr[j] = fmaf(float((cr >> (4 * j)) & 0xFu), s, z);
#pragma unroll
      for (int n = 0; n < NQ; ++n) {
        const int l = lq[n];
        float w = p_sm[warp][tt][n];
        if (l != L - 1) w *= half_bits_to_float(a.cache.alpha[1][l][slot * a.cap + tv]);
#pragma unroll
        for (int j = 0; j < P; ++j) acc_ref[n][j] = fmaf(w, vr[j], acc_ref[n][j]);
      }
      for (int l = l_first; l <= l_last; ++l) {
        if (l == L - 1) continue;
        const int bits = a.res_bits[l];
        const int row = D * bits / 8;
        const uint8_t* rc = a.cache.res_codes[1][l] + slot * a.cap * row;
        const uint32_t ce = load_v_lane_codes<P>(rc, tv, bits, lane);
        half2_bits(*reinterpret_cast<const uint32_t*>(a.cache.res_meta[1][l] +
                                                      (slot * a.cap + tv) * 2 * NG + 2 * grp),
                   s, z);
        const uint32_t mask = (1u << bits) - 1u;
        float e[P];
#pragma unroll
        for (int j = 0; j < P; ++j) e[j] = fmaf(float((ce >> (bits * j)) & mask), s, z);
#pragma unroll
        for (int n = 0; n < NQ; ++n) {
          if (lq[n] != l) continue;
          const float w = p_sm[warp][tt][n];
#pragma unroll
          for (int j = 0; j < P; ++j) acc_res[n][j] = fmaf(w, e[j], acc_res[n][j]);
        }
      }
    }
    __syncwarp();
  }

  // ---------------- merge the warps, write this split's partials ----------------
#pragma unroll
  for (int n = 0; n < NQ; ++n) {
    const float lsum = warp_sum(l_lane[n]);
    if (lane == 0) {
      m_sm[warp][n] = m_run[n];
      l_sm[warp][n] = lsum;
    }
#pragma unroll
    for (int j = 0; j < P; ++j) {
      acc_sm[warp][n][0][lane * P + j] = acc_ref[n][j];
      acc_sm[warp][n][1][lane * P + j] = acc_res[n][j];
    }
  }
  __syncthreads();
  const int rec = 2 + 2 * D;
  for (int n = warp; n < a.nq; n += kWarps) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, m_sm[w][n]);
    float f[kWarps];
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      f[w] = (m_sm[w][n] == -INFINITY) ? 0.f : exp2f(m_sm[w][n] - M);
      lt += f[w] * l_sm[w][n];
    }
    const int qn = a.q0 + n;
    const int li = qn / a.g, gi = qn % a.g;
    const int hq = h * a.g + gi;
    float* out = a.ws + (((int64_t(b) * a.Hq + hq) * a.loop_count + li) * a.n_splits + split) * rec;
    if (lane == 0) {
      out[0] = M;
      out[1] = lt;
    }
    for (int i = lane; i < 2 * D; i += 32) {
      const int part = i / D, ch = i % D;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += f[w] * acc_sm[w][n][part][ch];
      out[2 + i] = v;
    }
  }
}

// One warp per (b, query head, loop in the call): merge the split partials, add the
// current token's BF16 K/V, undo the rotation on the residual accumulator, store bf16.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const int8_t* __restrict__ v_signs,
                                                      const uint16_t* __restrict__ q,
                                                      const uint16_t* __restrict__ pending,
                                                      const float* __restrict__ ws,
                                                      uint16_t* __restrict__ out, int B, int Hq,
                                                      int H, int loop_count, int n_splits,
                                                      float scale_log2) {
  constexpr int P = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t wid = int64_t(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (wid >= int64_t(B) * Hq * loop_count) return;
  const int li = int(wid % loop_count);
  const int hq = int((wid / loop_count) % Hq);
  const int b = int(wid / (int64_t(loop_count) * Hq));
  const int h = hq / (Hq / H);
  const int rec = 2 + 2 * D;
  const float* part = ws + wid * n_splits * rec;

  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, part[s * rec]);
  float ps = -INFINITY;
  float kp[P], vp[P];
  if (pending) {
    const uint16_t* qp = q + wid * D + lane * P;
    const uint16_t* kpp = pending + ((int64_t(b) * 2 + 0) * loop_count + li) * H * D +
                          int64_t(h) * D + lane * P;
    const uint16_t* vpp = pending + ((int64_t(b) * 2 + 1) * loop_count + li) * H * D +
                          int64_t(h) * D + lane * P;
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      kp[j] = bf16_bits_to_float(kpp[j]);
      vp[j] = bf16_bits_to_float(vpp[j]);
      dot = fmaf(bf16_bits_to_float(qp[j]) * scale_log2, kp[j], dot);
    }
    ps = warp_sum(dot);
    M = fmaxf(M, ps);
  }
  float ar[P], ae[P];
#pragma unroll
  for (int j = 0; j < P; ++j) ar[j] = ae[j] = 0.f;
  float ell = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const float ms = part[s * rec];
      if (ms == -INFINITY) continue;
      const float f = exp2f(ms - M);
      ell += f * part[s * rec + 1];
#pragma unroll
      for (int j = 0; j < P; ++j) {
        ar[j] = fmaf(f, part[s * rec + 2 + lane * P + j], ar[j]);
        ae[j] = fmaf(f, part[s * rec + 2 + D + lane * P + j], ae[j]);
      }
    }
    if (pending) {
      const float f = exp2f(ps - M);
      ell += f;
#pragma unroll
      for (int j = 0; j < P; ++j) ar[j] = fmaf(f, vp[j], ar[j]);
    }
  }
  if (v_signs) {  // R^T y = signs * (H y) / sqrt(d)
    warp_fwht<P>(ae, lane);
    const int8_t* sg = v_signs + int64_t(h) * D + lane * P;
    const float inv_sqrt_d = (D == 128) ? 0.08838834764831845f : 0.125f;
#pragma unroll
    for (int j = 0; j < P; ++j) ar[j] = fmaf(ae[j] * inv_sqrt_d, float(sg[j]), ar[j]);
  }
  const float inv = ell > 0.f ? 1.f / ell : 0.f;
  uint16_t* o = out + wid * D + lane * P;
#pragma unroll
  for (int j = 0; j < P; ++j) o[j] = float_to_bf16_bits(ar[j] * inv);
}

}  // namespace

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

SplitPlan plan_splits(const rq_shape& s, int loop_count, int max_ctx) {
  (void)loop_count;
  SplitPlan p;
  const int units = s.batch * s.n_kv_heads;
  const int target = device_sm_count() * 8;
  int max_splits = (max_ctx + 2 * kCtaTokens - 1) / (2 * kCtaTokens);
  if (max_splits < 1) max_splits = 1;
  int splits = (target + units - 1) / units;
  splits = splits < 1 ? 1 : (splits > max_splits ? max_splits : splits);
  if (splits > 256) splits = 256;
  int per = (max_ctx + splits - 1) / splits;
  per = ((per + kCtaTokens - 1) / kCtaTokens) * kCtaTokens;
  if (per < kCtaTokens) per = kCtaTokens;
  p.tokens_per_split = per;
  p.n_splits = max_ctx > 0 ? (max_ctx + per - 1) / per : 1;
  return p;
}

size_t partial_floats(const rq_shape& s) { return size_t(2 + 2 * s.head_dim); }

cudaError_t launch_rq_decode(const rq_shape& s, const rq_cache& cache, const uint16_t* q,
                             int loop_begin, int loop_count, const uint16_t* pending,
                             const int32_t* ctx_lens, int max_ctx, uint16_t* out, float* ws,
                             cudaStream_t stream) {
  const SplitPlan plan = plan_splits(s, loop_count, max_ctx);
  DecodeArgs a;
  a.cache = cache;
  a.q = q;
  a.ctx_lens = ctx_lens;
  a.ws = ws;
  a.B = s.batch;
  a.Hq = s.n_q_heads;
  a.H = s.n_kv_heads;
  a.L = s.n_loops;
  a.cap = s.capacity;
  a.g = s.n_q_heads / s.n_kv_heads;
  a.loop_begin = loop_begin;
  a.loop_count = loop_count;
  a.n_splits = plan.n_splits;
  a.tokens_per_split = plan.tokens_per_split;
  const float scale = s.softmax_scale > 0.f ? s.softmax_scale : 1.0f / sqrtf(float(s.head_dim));
  a.scale_log2 = scale * kLog2e;
  for (int l = 0; l < RQ_MAX_LOOPS; ++l) a.res_bits[l] = s.res_bits[l];
  dim3 grid(plan.n_splits, s.n_kv_heads, s.batch);
  cudaError_t e;
  {  // query blocks of at most 8 queries per kv-head
    const int nq_total = a.g * loop_count;
    for (int q0 = 0; q0 < nq_total; q0 += 8) {
      DecodeArgs b = a;
      b.q0 = q0;
      b.nq = min(8, nq_total - q0);
      if (s.head_dim == 128) {
        if (b.nq == 1) rq_split_kernel<128, 1><<<grid, kWarps * 32, 0, stream>>>(b);
        else if (b.nq == 2) rq_split_kernel<128, 2><<<grid, kWarps * 32, 0, stream>>>(b);
        else if (b.nq <= 4) rq_split_kernel<128, 4><<<grid, kWarps * 32, 0, stream>>>(b);
        else rq_split_kernel<128, 8><<<grid, kWarps * 32, 0, stream>>>(b);
      } else {
        if (b.nq == 1) rq_split_kernel<64, 1><<<grid, kWarps * 32, 0, stream>>>(b);
        else if (b.nq == 2) rq_split_kernel<64, 2><<<grid, kWarps * 32, 0, stream>>>(b);
        else if (b.nq <= 4) rq_split_kernel<64, 4><<<grid, kWarps * 32, 0, stream>>>(b);
        else rq_split_kernel<64, 8><<<grid, kWarps * 32, 0, stream>>>(b);
      }
    }
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  return launch_combine(s, cache.rot_signs[1], q, loop_count, pending, plan.n_splits, out, ws,
                        stream);
}

cudaError_t launch_combine(const rq_shape& s, const int8_t* v_signs, const uint16_t* q,
                           int loop_count, const uint16_t* pending, int n_splits,
                           uint16_t* out, const float* ws, cudaStream_t stream) {
  const int64_t warps = int64_t(s.batch) * s.n_q_heads * loop_count;
  const unsigned blocks = unsigned((warps + 3) / 4);
  const float scale = s.softmax_scale > 0.f ? s.softmax_scale : 1.0f / sqrtf(float(s.head_dim));
  if (s.head_dim == 128)
    combine_kernel<128><<<blocks, 128, 0, stream>>>(v_signs, q, pending, ws, out, s.batch,
                                                    s.n_q_heads, s.n_kv_heads, loop_count,
                                                    n_splits, scale * kLog2e);
  else
    combine_kernel<64><<<blocks, 128, 0, stream>>>(v_signs, q, pending, ws, out, s.batch,
                                                   s.n_q_heads, s.n_kv_heads, loop_count,
                                                   n_splits, scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace rq
