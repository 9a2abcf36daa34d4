// Synthetic looped K/V states and queries written straight into device memory.
// Philox4x32-10 (Salmon et al., SC'11) + correctly rounded fp32 operations: the values
// equal, bit for bit, those of the host-side generator used by the CPU oracle.
#include "../../include/rq_synth.h"
#include "rq_common.cuh"

namespace rq {
namespace {

constexpr int kFieldBase = 1, kFieldNoise = 2, kFieldU = 3, kFieldQuery = 4;

struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                     uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return {c0, c1, c2, c3};
}

__device__ __forceinline__ uint32_t c2_of(int h, int kv, int l, int i) {
  return (uint32_t(h) << 16) | (uint32_t(kv) << 15) | (uint32_t(l) << 8) | uint32_t(i);
}

__device__ __forceinline__ uint32_t c3_of(int field, int layer, int sub) {
  return (uint32_t(field) << 24) | ((uint32_t(layer) & 0xFFFFu) << 8) | (uint32_t(sub) & 0xFFu);
}

__device__ __forceinline__ int fields10(uint32_t w) {
  return int(w & 1023u) + int((w >> 10) & 1023u) + int((w >> 20) & 1023u);
}

__device__ __forceinline__ float normal(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                        uint32_t k0, uint32_t k1) {
  U4 r = philox(c0, c1, c2, c3, k0, k1);
  int s = fields10(r.x) + fields10(r.y) + fields10(r.z) + fields10(r.w);
  return __fmul_rn(float(s - 6138), 1.0f / 1024.0f);  // exact
}

__global__ void synth_states_kernel(rq_synth_params p, uint16_t* __restrict__ out,
                                    int64_t s0, int64_t s1, int64_t s2, int64_t s3, int64_t s4,
                                    int b0, int nb, int t0, int nt, int l0, int nl) {
  const int d = p.head_dim;
  const int H = p.n_kv_heads;
  const uint32_t k0 = uint32_t(p.seed), k1 = uint32_t(p.seed >> 32);
  // one thread per (b, t, kv, h, i); loops inside (base is shared by the loops)
  const int64_t n = int64_t(nb) * nt * 2 * H * d;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < n;
       e += int64_t(gridDim.x) * blockDim.x) {
    int64_t r = e;
    const int i = int(r % d); r /= d;
    const int h = int(r % H); r /= H;
    const int kv = int(r % 2); r /= 2;
    const int tt = int(r % nt); r /= nt;
    const int bb = int(r);
    const uint32_t t = uint32_t(t0 + tt), b = uint32_t(b0 + bb);
    float base;
    const uint32_t c2b = c2_of(h, kv, 0, i);
    if (p.dist == 1) {
      float z0 = normal(t, b, c2b, c3_of(kFieldBase, p.layer, 0), k0, k1);
      float z1 = normal(t, b, c2b, c3_of(kFieldBase, p.layer, 1), k0, k1);
      float z2 = normal(t, b, c2b, c3_of(kFieldBase, p.layer, 2), k0, k1);
      float z3 = normal(t, b, c2b, c3_of(kFieldBase, p.layer, 3), k0, k1);
      float chi = __fadd_rn(__fadd_rn(__fmul_rn(z1, z1), __fmul_rn(z2, z2)), __fmul_rn(z3, z3));
      float v = __fdiv_rn(chi, 3.0f);
      v = fmaxf(v, 0.0009765625f);  // 2^-10
      base = __fdiv_rn(z0, __fsqrt_rn(v));
    } else {
      base = normal(t, b, c2b, c3_of(kFieldBase, p.layer, 0), k0, k1);
    }
    if (p.n_outliers > 0) {
      const int32_t* ot = p.outlier_table + (int64_t(h) * 2 + kv) * p.n_outliers;
      for (int o = 0; o < p.n_outliers; ++o)
        if (ot[o] == i) base = __fmul_rn(base, p.outlier_mult);
    }
    for (int ll = 0; ll < nl; ++ll) {
      const int l = l0 + ll;
      U4 wu = philox(t, b, c2_of(h, kv, l, 0), c3_of(kFieldU, p.layer, 0), k0, k1);
      float u01 = __fmul_rn(__fadd_rn(float(wu.x >> 8), 0.5f), 5.9604644775390625e-8f);
      float u = __fadd_rn(0.8f, __fmul_rn(0.4f, u01));
      float nz = normal(t, b, c2_of(h, kv, l, i), c3_of(kFieldNoise, p.layer, 0), k0, k1);
      float x = __fadd_rn(__fmul_rn(u, base), __fmul_rn(p.sigma[l], nz));
      out[int64_t(bb) * s0 + int64_t(tt) * s1 + int64_t(kv) * s2 + int64_t(ll) * s3 +
          int64_t(h) * s4 + i] = float_to_bf16_bits(x);
    }
  }
}

__global__ void synth_queries_kernel(rq_synth_params p, uint16_t* __restrict__ out, int Hq,
                                     int b0, int nb, int l0, int nl, int step) {
  const int d = p.head_dim;
  const uint32_t k0 = uint32_t(p.seed), k1 = uint32_t(p.seed >> 32);
  const int64_t n = int64_t(nb) * Hq * nl * d;
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < n;
       e += int64_t(gridDim.x) * blockDim.x) {
    int64_t r = e;
    const int i = int(r % d); r /= d;
    const int ll = int(r % nl); r /= nl;
    const int qh = int(r % Hq); r /= Hq;
    const int bb = int(r);
    float z = normal(uint32_t(step), uint32_t(b0 + bb), c2_of(qh, 0, l0 + ll, i),
                     c3_of(kFieldQuery, p.layer, 0), k0, k1);
    out[e] = float_to_bf16_bits(z);
  }
}

int grid_for(int64_t n, int threads) {
  int64_t g = (n + threads - 1) / threads;
  if (g > (1 << 20)) g = 1 << 20;
  return int(g < 1 ? 1 : g);
}

}  // namespace
}  // namespace rq

extern "C" rq_status rq_synth_states(const rq_synth_params* p, uint16_t* out,
                                     const int64_t strides[5], int32_t b0, int32_t nb,
                                     int32_t t0, int32_t nt, int32_t l0, int32_t nl,
                                     void* stream) {
  if (!p || !out || !strides) return RQ_ERR_INVALID_ARG;
  if (p->head_dim <= 0 || p->head_dim > 256 || p->n_kv_heads <= 0 || p->n_kv_heads > 65535)
    return RQ_ERR_INVALID_ARG;
  if (nb < 0 || nt < 0 || nl < 0 || b0 < 0 || t0 < 0 || l0 < 0 || l0 + nl > RQ_MAX_LOOPS)
    return RQ_ERR_INVALID_ARG;
  if (p->n_outliers < 0 || p->n_outliers > 8 || (p->n_outliers > 0 && !p->outlier_table))
    return RQ_ERR_INVALID_ARG;
  for (int k = 0; k < 5; ++k)
    if (strides[k] < 0) return RQ_ERR_INVALID_ARG;
  const int64_t n = int64_t(nb) * nt * 2 * p->n_kv_heads * p->head_dim;
  if (n == 0 || nl == 0) return RQ_OK;
  rq::synth_states_kernel<<<rq::grid_for(n, 256), 256, 0, (cudaStream_t)stream>>>(
      *p, out, strides[0], strides[1], strides[2], strides[3], strides[4], b0, nb, t0, nt,
      l0, nl);
  return cudaGetLastError() == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

extern "C" rq_status rq_synth_queries(const rq_synth_params* p, uint16_t* out,
                                      int32_t n_q_heads, int32_t b0, int32_t nb, int32_t l0,
                                      int32_t nl, int32_t step, void* stream) {
  if (!p || !out || n_q_heads <= 0 || n_q_heads > 65535 || nb < 0 || nl < 0 || b0 < 0 ||
      l0 < 0 || l0 + nl > RQ_MAX_LOOPS || p->head_dim <= 0 || p->head_dim > 256)
    return RQ_ERR_INVALID_ARG;
  const int64_t n = int64_t(nb) * n_q_heads * nl * p->head_dim;
  if (n == 0) return RQ_OK;
  rq::synth_queries_kernel<<<rq::grid_for(n, 256), 256, 0, (cudaStream_t)stream>>>(
      *p, out, n_q_heads, b0, nb, l0, nl, step);
  return cudaGetLastError() == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}
