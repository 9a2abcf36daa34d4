// Comparison kernel: split-KV decode attention over an uncompressed BF16 per-loop cache
// [B][Hkv][L][cap][d], same split plan, partial format and combine as the packed path.
#include "rq_common.cuh"
#include "rq_kernels.h"

namespace rq {
namespace {

constexpr int kWarps = 4;
constexpr int kChunk = 32;
constexpr int kCtaTokens = kWarps * kChunk;

struct Bf16Args {
  const uint16_t* k;
  const uint16_t* v;
  const uint16_t* q;
  const int32_t* ctx_lens;
  float* ws;
  int B, Hq, H, L, cap, g, loop_begin, loop_count, n_splits, tokens_per_split;
  float scale_log2;
};

__device__ __forceinline__ void bf16x8(const uint4 r, float (&f)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

// grid (splits, Hkv, B * loop_count); NQ = g query heads of one loop.
template <int D, int NQ>
__global__ void __launch_bounds__(kWarps * 32) bf16_split_kernel(Bf16Args a) {
  constexpr int P = D / 32;
  __shared__ __align__(16) float q_sm[NQ][D];
  __shared__ float p_sm[kWarps][kChunk][NQ];
  __shared__ float m_sm[kWarps][NQ], l_sm[kWarps][NQ];
  __shared__ __align__(16) float acc_sm[kWarps][NQ][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, h = blockIdx.y;
  const int b = blockIdx.z / a.loop_count, li = blockIdx.z % a.loop_count;
  const int l = a.loop_begin + li;
  const int ctx = min(a.ctx_lens[b], a.cap);
  const int t_begin = split * a.tokens_per_split;
  const int t_end = min(ctx, t_begin + a.tokens_per_split);

  for (int n = warp; n < NQ; n += kWarps) {
    const int gi = min(n, a.g - 1);
    const uint16_t* qp = a.q + ((int64_t(b) * a.Hq + h * a.g + gi) * a.loop_count + li) * D;
    for (int i = lane; i < D; i += 32) q_sm[n][i] = bf16_bits_to_float(qp[i]) * a.scale_log2;
  }
  __syncthreads();

  const int64_t base = ((int64_t(b) * a.H + h) * a.L + l) * int64_t(a.cap) * D;
  const uint16_t* kp = a.k + base;
  const uint16_t* vp = a.v + base;

  float m_run[NQ], l_lane[NQ], acc[NQ][P];
#pragma unroll
  for (int n = 0; n < NQ; ++n) {
    m_run[n] = -INFINITY;
    l_lane[n] = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) acc[n][j] = 0.f;
  }

  for (int c0 = t_begin + warp * kChunk; c0 < t_end; c0 += kCtaTokens) {
    const int t = c0 + lane;
    const bool valid = t < t_end;
    const int tl = valid ? t : c0;
    float sc[NQ];
#pragma unroll
    for (int n = 0; n < NQ; ++n) sc[n] = 0.f;
    const uint4* krow = reinterpret_cast<const uint4*>(kp + int64_t(tl) * D);
#pragma unroll 4
    for (int c = 0; c < D / 8; ++c) {
      float f[8];
      bf16x8(krow[c], f);
#pragma unroll
      for (int n = 0; n < NQ; ++n) {
        const float4 q0 = *reinterpret_cast<const float4*>(&q_sm[n][8 * c]);
        const float4 q1 = *reinterpret_cast<const float4*>(&q_sm[n][8 * c + 4]);
        float s = sc[n];
        s = fmaf(f[0], q0.x, s);
        s = fmaf(f[1], q0.y, s);
        s = fmaf(f[2], q0.z, s);
        s = fmaf(f[3], q0.w, s);
        s = fmaf(f[4], q1.x, s);
        s = fmaf(f[5], q1.y, s);
        s = fmaf(f[6], q1.z, s);
        s = fmaf(f[7], q1.w, s);
        sc[n] = s;
      }
    }
#pragma unroll
    for (int n = 0; n < NQ; ++n) {
      const float score = valid ? sc[n] : -INFINITY;
      const float m_new = fmaxf(m_run[n], warp_max(score));
      const float corr = (m_run[n] == -INFINITY) ? 0.f : exp2f(m_run[n] - m_new);
      const float p = valid ? exp2f(score - m_new) : 0.f;
      l_lane[n] = l_lane[n] * corr + p;
#pragma unroll
      for (int j = 0; j < P; ++j) acc[n][j] *= corr;
      m_run[n] = m_new;
      p_sm[warp][lane][n] = p;
    }
    __syncwarp();
    const int nvalid = min(kChunk, t_end - c0);
    for (int tt = 0; tt < nvalid; ++tt) {
      const uint16_t* vr = vp + int64_t(c0 + tt) * D + lane * P;
      float vv[P];
      if (P == 4) {
        const uint2 r = *reinterpret_cast<const uint2*>(vr);
        vv[0] = __uint_as_float(r.x << 16);
        vv[1] = __uint_as_float(r.x & 0xFFFF0000u);
        vv[2 % P] = __uint_as_float(r.y << 16);
        vv[3 % P] = __uint_as_float(r.y & 0xFFFF0000u);
      } else {
        const uint32_t r = *reinterpret_cast<const uint32_t*>(vr);
        vv[0] = __uint_as_float(r << 16);
        vv[1 % P] = __uint_as_float(r & 0xFFFF0000u);
      }
#pragma unroll
      for (int n = 0; n < NQ; ++n) {
        const float w = p_sm[warp][tt][n];
#pragma unroll
        for (int j = 0; j < P; ++j) acc[n][j] = fmaf(w, vv[j], acc[n][j]);
      }
    }
    __syncwarp();
  }

#pragma unroll
  for (int n = 0; n < NQ; ++n) {
    const float lsum = warp_sum(l_lane[n]);
    if (lane == 0) {
      m_sm[warp][n] = m_run[n];
      l_sm[warp][n] = lsum;
    }
#pragma unroll
    for (int j = 0; j < P; ++j) acc_sm[warp][n][lane * P + j] = acc[n][j];
  }
  __syncthreads();
  const int rec = int(partial_floats_d(D));
  for (int n = warp; n < a.g; n += kWarps) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, m_sm[w][n]);
    float f[kWarps], lt = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      f[w] = (m_sm[w][n] == -INFINITY) ? 0.f : exp2f(m_sm[w][n] - M);
      lt += f[w] * l_sm[w][n];
    }
    const int hq = h * a.g + n;
    float* out = a.ws + (((int64_t(b) * a.Hq + hq) * a.loop_count + li) * a.n_splits + split) * rec;
    if (lane == 0) {
      out[0] = M;
      out[1] = lt;
    }
    for (int i = lane; i < D; i += 32) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += f[w] * acc_sm[w][n][i];
      out[4 + i] = v;
      out[4 + D + i] = 0.f;
    }
  }
}

template <int D>
void launch_d(const Bf16Args& a, dim3 grid, cudaStream_t stream) {
  if (a.g == 1) bf16_split_kernel<D, 1><<<grid, kWarps * 32, 0, stream>>>(a);
  else if (a.g == 2) bf16_split_kernel<D, 2><<<grid, kWarps * 32, 0, stream>>>(a);
  else if (a.g <= 4) bf16_split_kernel<D, 4><<<grid, kWarps * 32, 0, stream>>>(a);
  else bf16_split_kernel<D, 8><<<grid, kWarps * 32, 0, stream>>>(a);
}

}  // namespace

cudaError_t launch_bf16_decode(const rq_shape& s, const uint16_t* k, const uint16_t* v,
                               const uint16_t* q, int loop_begin, int loop_count,
                               const uint16_t* pending, const int32_t* ctx_lens, int max_ctx,
                               uint16_t* out, float* ws, cudaStream_t stream) {
  const SplitPlan plan = plan_splits_bf16(s, max_ctx);
  ws += kWsHeaderBytes / sizeof(float);
  Bf16Args a;
  a.k = k;
  a.v = v;
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
  dim3 grid(plan.n_splits, s.n_kv_heads, s.batch * loop_count);
  if (s.head_dim == 128)
    launch_d<128>(a, grid, stream);
  else
    launch_d<64>(a, grid, stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine(s, nullptr, q, loop_count, pending, plan.n_splits, out, ws, nullptr,
                        stream);
}

}  // namespace rq
