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

// Walsh-Hadamard transform (Sylvester order, unnormalised) of a d-vector spread over a
// warp: lane holds channels [lane*P, lane*P + P), P = d / 32 in {2, 4}.  Channel index
// bits below log2(P) are butterflied in registers, the rest across lanes.
template <int P>
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
  for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
    for (int j = 0; j < P; ++j) {
      float u = __shfl_xor_sync(RQ_FULL_MASK, v[j], m);
      v[j] = (lane & m) ? (u - v[j]) : (v[j] + u);
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

}  // namespace rq
