// Shared device helpers of the librq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rq.h"

#define RQ_FULL_MASK 0xffffffffu

namespace rq {

constexpr int kGroup = 32;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ uint16_t float_to_half_bits(float f) {
  return __half_as_ushort(__float2half_rn(f));
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(RQ_FULL_MASK, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(RQ_FULL_MASK, v, o));
  return v;
}

// Walsh-Hadamard transform (Sylvester order, unnormalised) of a d-vector spread over LANES
// lanes (a warp, or each half of it): lane i of the group holds channels [i*P, i*P + P),
// P = d / LANES.  Channel index bits below log2(P) are butterflied in registers, the rest
// across lanes, lowest bit first.
template <int P, int LANES = 32>
__device__ __forceinline__ void warp_fwht(float (&v)[P], int lane) {
#pragma unroll
  for (int h = 1; h < P; h <<= 1) {
#pragma unroll
    for (int j = 0; j < P; ++j) {
      if ((j & h) == 0) {
        float a = v[j], b = v[j + h];
        v[j] = a + b;
        v[j + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < LANES; m <<= 1) {
    // the lane holding index bit m takes u - v, its partner v + u: one fused u + sign * v
    // (sign * v is exact, so the result is the same single rounding)
    const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const float u = __shfl_xor_sync(RQ_FULL_MASK, v[j], m);
      v[j] = fmaf(sgn, v[j], u);
    }
  }
}

// XOR applied to the 16-bit unit index in row pair p of a V code array whose rows hold
// `units` 16-bit units: it spreads the pairs a fragment load touches over distinct banks.
__host__ __device__ __forceinline__ int v_unit_swizzle(int64_t p, int units) {
  return units == 32 ? int(8 * (p & 3)) : (units == 16 ? int(8 * ((p >> 1) & 1)) : 0);
}

// Byte offset of natural byte k of token t's row in a V code array stored in token pairs:
// in pair p = t/2 the 32-bit word at position u ^ swizzle(p) holds 16-bit unit u = k/2 of
// token 2p (low half) and of token 2p+1 (high half).  Relative to the (b, h) slot base.
__device__ __forceinline__ int64_t vpair_offset(int64_t t, int k, int row_bytes) {
  const int64_t p = t >> 1;
  const int u = (k >> 1) ^ v_unit_swizzle(p, row_bytes >> 1);
  return p * (2 * row_bytes) + u * 4 + (t & 1) * 2 + (k & 1);
}

// Byte offset, within a K code row, of natural byte k: words are group-interleaved (the
// j-th word of every 32-channel group adjacent), word w -> (w % bits) * (d/32) + w / bits.
__device__ __forceinline__ int k_row_offset(int k, int bits, int ng) {
  const int w = k >> 2;
  return ((w % bits) * ng + w / bits) * 4 + (k & 3);
}

// Split combine of one query column by one warp: merge the split partial records (m, l, two
// pad floats, acc_ref[D], acc_res[D]), add the current token's BF16 K/V (kp, vp rows, or
// null), undo the rotation of the residual accumulator (R^T y = signs * (H y) / sqrt(d);
// signs of the column's kv-head, or null when there is no residual part), store bf16.
// `failed` (a split gave up) makes the output NaN.
template <int D>
__device__ __forceinline__ void combine_column(const float* part, int n_splits, const uint16_t* qp,
                                               const uint16_t* kpp, const uint16_t* vpp,
                                               const int8_t* sg, float scale_log2, bool failed,
                                               uint16_t* o, int lane) {
  constexpr int P = D / 32;
  constexpr int rec = 4 + 2 * D;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, part[s * rec]);
  float ps = -INFINITY;
  float vp[P];
  if (kpp) {
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      vp[j] = bf16_bits_to_float(vpp[lane * P + j]);
      dot = fmaf(bf16_bits_to_float(qp[lane * P + j]) * scale_log2,
                 bf16_bits_to_float(kpp[lane * P + j]), dot);
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
        ar[j] = fmaf(f, part[s * rec + 4 + lane * P + j], ar[j]);
        ae[j] = fmaf(f, part[s * rec + 4 + D + lane * P + j], ae[j]);
      }
    }
    if (kpp) {
      const float f = exp2f(ps - M);
      ell += f;
#pragma unroll
      for (int j = 0; j < P; ++j) ar[j] = fmaf(f, vp[j], ar[j]);
    }
  }
  if (sg) {
    warp_fwht<P>(ae, lane);
    const float inv_sqrt_d = (D == 128) ? 0.08838834764831845f : 0.125f;
#pragma unroll
    for (int j = 0; j < P; ++j) ar[j] = fmaf(ae[j] * inv_sqrt_d, float(sg[lane * P + j]), ar[j]);
  }
  float inv = ell > 0.f ? 1.f / ell : 0.f;
  if (failed) inv = __int_as_float(0x7fc00000);
#pragma unroll
  for (int j = 0; j < P; ++j) o[lane * P + j] = float_to_bf16_bits(ar[j] * inv);
}

}  // namespace rq
