// ResidualQuant encode: runs once the token's final loop has finished (deferred write,
// rit.work summary "How each pass's KV cache is reconstructed").  VL lanes encode one
// (sequence, new token, kv-head, K/V): the final loop's state becomes the INT4 reference,
// every other loop a least-squares-scaled, Hadamard-rotated 2- or 4-bit residual.  Large
// calls (bulk prefill) put K and V of a token in the two halves of a warp (VL 16: fewer
// shuffle stages and instructions per vector); small ones (the per-step append) give a
// vector a whole warp (VL 32: the shortest dependency chain per vector).
#include "rq_common.cuh"
#include "rq_kernels.h"

namespace rq {
namespace {

struct EncodeArgs {
  uint8_t* data;         // tile records of the packed cache
  int64_t rec_bytes;     // bytes of one record
  const int8_t* rot_signs[2];
  const uint16_t* kv_new;
  int64_t sb, st, skv, sl, sh;  // element strides of kv_new
  const int32_t* positions;
  int32_t pos_begin;
  int32_t n_new;
  int32_t B, H, L, cap;
  int8_t res_bits[RQ_MAX_LOOPS];
  const int32_t* bt;     // block table of a paged cache, or null
  int32_t max_pages, n_pages;
  int32_t vec;           // kv_new rows allow one vector load of a lane's channels
  int32_t alpha_mode;    // 0: least-squares a_l (the method); 1: a = 1; 2: a = 0 (ablations)
};

// Sum over the VL lanes of a vector.
template <int VL>
__device__ __forceinline__ float vec_sum(float v) {
#pragma unroll
  for (int o = VL / 2; o > 0; o >>= 1) v += __shfl_xor_sync(RQ_FULL_MASK, v, o);
  return v;
}

// Group min / max over the lanes that share a 32-channel group (LPG lanes).
template <int LPG>
__device__ __forceinline__ void group_minmax(float& mn, float& mx) {
#pragma unroll
  for (int o = 1; o < LPG; o <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(RQ_FULL_MASK, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(RQ_FULL_MASK, mx, o));
  }
}

// Quantise the P channels this lane holds with (step, offset) from the group's min/max;
// returns the codes, writes the dequantised values into deq and the fp16 pair into s_h/z_h.
template <int P, int LEVELS>
__device__ __forceinline__ void quantize_lane(const float (&v)[P], int (&c)[P], float (&deq)[P],
                                              uint16_t& s_bits, uint16_t& z_bits) {
  constexpr int LPG = kGroup / P;
  float mn = v[0], mx = v[0];
#pragma unroll
  for (int j = 1; j < P; ++j) {
    mn = fminf(mn, v[j]);
    mx = fmaxf(mx, v[j]);
  }
  group_minmax<LPG>(mn, mx);
  const float s = __fdiv_rn(__fsub_rn(mx, mn), float(LEVELS));
  s_bits = float_to_half_bits(s);
  z_bits = float_to_half_bits(mn);
  const float s_h = half_bits_to_float(s_bits);
  const float z_h = half_bits_to_float(z_bits);
  // (x - z) / s correctly rounded from the correctly rounded reciprocal y of s: q = RN(n y),
  // then one correction RN(q + RN(n - q s) y) (Markstein's quotient correction, which gives
  // the correctly rounded quotient when y is the correctly rounded 1/s); s is an fp16 value
  // > 0 and n is bounded, so no intermediate leaves the normal fp32 range
  const float y = s_h > 0.0f ? __frcp_rn(s_h) : 0.0f;
#pragma unroll
  for (int j = 0; j < P; ++j) {
    float qv = 0.0f;
    if (s_h > 0.0f) {
      const float n = __fsub_rn(v[j], z_h);
      const float q0 = __fmul_rn(n, y);
      const float rem = __fmaf_rn(-q0, s_h, n);
      qv = rintf(__fmaf_rn(rem, y, q0));
      qv = fminf(fmaxf(qv, 0.0f), float(LEVELS));
    }
    c[j] = int(qv);
    deq[j] = fmaf(qv, s_h, z_h);
  }
}

// Store the packed bits of the P channels of lane `lane` (of the vector's lanes), the
// natural row's bytes [lane * BITS * P / 8, ...): 8, 16 or 32 bits per lane.  K rows are
// group-interleaved (NG groups of 32 channels); V rows go to the token-pair layout.
template <int P, int BITS, int NG>
__device__ __forceinline__ void store_codes(uint8_t* slot, int64_t tok, int row_bytes, bool is_v,
                                            const int (&c)[P], int lane) {
  uint32_t w = 0;
#pragma unroll
  for (int j = 0; j < P; ++j) w |= uint32_t(c[j]) << (BITS * j);
  constexpr int LANE_BITS = BITS * P;
  static_assert(LANE_BITS == 8 || LANE_BITS == 16 || LANE_BITS == 32, "lane bits");
  if constexpr (LANE_BITS == 8) {
    const int k = lane;
    int64_t off = is_v ? vpair_offset(tok, k, row_bytes)
                       : tok * row_bytes + k_row_offset(k, BITS, NG);
    slot[off] = uint8_t(w);
  } else if constexpr (LANE_BITS == 16) {  // one aligned 16-bit unit
    const int k = 2 * lane;
    int64_t off = is_v ? vpair_offset(tok, k, row_bytes)
                       : tok * row_bytes + k_row_offset(k, BITS, NG);
    *reinterpret_cast<uint16_t*>(slot + off) = uint16_t(w);
  } else {  // 32 bits: one K word, or two 16-bit units of a V token pair
    const int k = 4 * lane;
    if (is_v) {
      *reinterpret_cast<uint16_t*>(slot + vpair_offset(tok, k, row_bytes)) = uint16_t(w);
      *reinterpret_cast<uint16_t*>(slot + vpair_offset(tok, k + 2, row_bytes)) = uint16_t(w >> 16);
    } else {
      *reinterpret_cast<uint32_t*>(slot + tok * row_bytes + k_row_offset(k, BITS, NG)) = w;
    }
  }
}

template <int D, int VL>
__global__ void __launch_bounds__(128, 8) encode_kernel(EncodeArgs a) {
  constexpr int P = D / VL;         // channels per lane
  constexpr int LPG = kGroup / P;   // lanes per 32-channel group
  constexpr int NG = D / kGroup;
  const int lane = threadIdx.x & 31;
  const int hl = lane & (VL - 1);   // lane within the vector
  // vectors (sequence, token, kv-head, K/V), K/V fastest: a warp's halves (VL 16) hold the
  // K and V states of one token and kv-head
  const int64_t vid = (int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * (32 / VL) +
                      lane / VL;
  const int64_t total = int64_t(a.B) * a.n_new * a.H * 2;
  if (vid >= total) return;
  int64_t r = vid;
  const int kv = int(r % 2); r /= 2;
  const int h = int(r % a.H); r /= a.H;
  const int j = int(r % a.n_new); r /= a.n_new;
  const int b = int(r);
  const int pos = a.positions ? a.positions[int64_t(b) * a.n_new + j] : a.pos_begin + j;
  if (pos < 0 || pos >= a.cap) return;
  const bool is_v = kv == 1;
  // the tile record holding the token (contiguous: record (b, h, pos / 64); paged: the
  // record of (page, h) of the 64-token page through the block table); the token is row
  // tok = pos % 64 of each of its sections
  int64_t rec_index;
  if (a.bt) {
    const int pg = a.bt[int64_t(b) * a.max_pages + (pos >> 6)];
    if (pg < 0 || pg >= a.n_pages) return;
    rec_index = int64_t(pg) * a.H + h;
  } else {
    rec_index = (int64_t(b) * a.H + h) * (a.cap / kTile) + (pos >> 6);
  }
  uint8_t* const rec = a.data + rec_index * a.rec_bytes;
  const int64_t tok = pos & 63;

  const uint16_t* src = a.kv_new + int64_t(b) * a.sb + int64_t(j) * a.st + int64_t(kv) * a.skv +
                        int64_t(h) * a.sh + hl * P;
  const int L = a.L;
  auto load = [&](int l, float (&v)[P]) {
    const uint16_t* p = src + int64_t(l) * a.sl;
    uint16_t e[P];
    if (a.vec) {   // one 16-byte (P 8) or 8-byte (P 4) load
      if constexpr (P == 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(p);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          e[2 * q] = uint16_t(u[q]);
          e[2 * q + 1] = uint16_t(u[q] >> 16);
        }
      } else {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        e[0] = uint16_t(w.x);
        e[1] = uint16_t(w.x >> 16);
        e[2] = uint16_t(w.y);
        e[3] = uint16_t(w.y >> 16);
      }
    } else {
#pragma unroll
      for (int q = 0; q < P; ++q) e[q] = p[q];
    }
#pragma unroll
    for (int q = 0; q < P; ++q) v[q] = bf16_bits_to_float(e[q]);
  };

  // ---- reference: the final loop, INT4 ----
  float x_ref[P], ref_hat[P];
  int c[P];
  load(L - 1, x_ref);
  uint16_t s_bits, z_bits;
  quantize_lane<P, 15>(x_ref, c, ref_hat, s_bits, z_bits);
  {
    // reference section: K codes, K meta, V codes, V meta (64 rows each)
    uint8_t* codes = rec + kv * (kTile * (D / 2) + kTile * NG * 4);
    store_codes<P, 4, NG>(codes, tok, D / 2, is_v, c, hl);
    if (hl % LPG == 0) {
      const int g = hl / LPG;
      uint8_t* meta = codes + kTile * (D / 2) + tok * (NG * 4) + g * 4;
      *reinterpret_cast<uint32_t*>(meta) = uint32_t(s_bits) | (uint32_t(z_bits) << 16);
    }
  }
  // <ref_hat, ref_hat> is shared by all loops
  float den = 0.f;
#pragma unroll
  for (int q = 0; q < P; ++q) den = fmaf(ref_hat[q], ref_hat[q], den);
  den = vec_sum<VL>(den);

  float sgn[P];
  {
    const int8_t* sp = a.rot_signs[kv] + int64_t(h) * D + hl * P;
#pragma unroll
    for (int q = 0; q < P; ++q) sgn[q] = float(sp[q]);
  }
  const float inv_sqrt_d = (D == 128) ? 0.08838834764831845f : 0.125f;

  for (int l = 0; l < L - 1; ++l) {
    float x[P];
    load(l, x);
    // least-squares scale against the dequantised reference
    float num = 0.f;
#pragma unroll
    for (int q = 0; q < P; ++q) num = fmaf(x[q], ref_hat[q], num);
    num = vec_sum<VL>(num);
    float alpha = den > 0.f ? __fdiv_rn(num, den) : 0.f;
    if (a.alpha_mode != 0) alpha = a.alpha_mode == 1 ? 1.f : 0.f;   // (ablation encodes)
    const uint16_t a_bits = float_to_half_bits(alpha);
    const float a_h = half_bits_to_float(a_bits);
    // loop l's section: K codes, K meta, K a, V codes, V meta, V a (64 rows each)
    const int bits = a.res_bits[l];
    const int row = D * bits / 8;
    uint8_t* const sec = rec + loop_section_offset(D, a.res_bits, l) +
                         kv * (kTile * row + kTile * NG * 4 + kTile * 2);
    if (hl == 0)
      *reinterpret_cast<uint16_t*>(sec + kTile * row + kTile * NG * 4 + tok * 2) = a_bits;
    // residual, rotation R r = H (signs * r) / sqrt(d)
    float y[P];
#pragma unroll
    for (int q = 0; q < P; ++q) y[q] = fmaf(-a_h, ref_hat[q], x[q]) * sgn[q];
    warp_fwht<P, VL>(y, hl);
#pragma unroll
    for (int q = 0; q < P; ++q) y[q] *= inv_sqrt_d;
    float deq[P];
    uint8_t* codes = sec;
    if (bits == 2) {
      quantize_lane<P, 3>(y, c, deq, s_bits, z_bits);
      store_codes<P, 2, NG>(codes, tok, row, is_v, c, hl);
    } else {
      quantize_lane<P, 15>(y, c, deq, s_bits, z_bits);
      store_codes<P, 4, NG>(codes, tok, row, is_v, c, hl);
    }
    if (hl % LPG == 0) {
      const int g = hl / LPG;
      uint8_t* meta = sec + kTile * row + tok * (NG * 4) + g * 4;
      *reinterpret_cast<uint32_t*>(meta) = uint32_t(s_bits) | (uint32_t(z_bits) << 16);
    }
  }
}

}  // namespace

cudaError_t launch_encode(const rq_shape& s, const rq_cache& cache, const rq_paging* paging,
                          const uint16_t* kv_new,
                          const int64_t strides[5], const int32_t* positions, int32_t pos_begin,
                          int32_t n_new, cudaStream_t stream, int alpha_mode) {
  EncodeArgs a;
  a.alpha_mode = alpha_mode;
  a.data = cache.data;
  a.rec_bytes = record_bytes(s);
  a.rot_signs[0] = cache.rot_signs[0];
  a.rot_signs[1] = cache.rot_signs[1];
  a.kv_new = kv_new;
  a.sb = strides[0];
  a.st = strides[1];
  a.skv = strides[2];
  a.sl = strides[3];
  a.sh = strides[4];
  a.positions = positions;
  a.pos_begin = pos_begin;
  a.n_new = n_new;
  a.B = s.batch;
  a.H = s.n_kv_heads;
  a.L = s.n_loops;
  a.cap = s.capacity;
  for (int l = 0; l < RQ_MAX_LOOPS; ++l) a.res_bits[l] = s.res_bits[l];
  a.bt = paging ? paging->block_table : nullptr;
  a.max_pages = paging ? paging->max_pages : 0;
  a.n_pages = paging ? paging->n_pages : 0;
  // vectors of the call; below a few per SM, a vector of d 128 gets a whole warp
  const int64_t vectors = int64_t(s.batch) * n_new * s.n_kv_heads * 2;
  const int vl = (s.head_dim == 128 && vectors < 64 * 152) ? 32 : 16;
  // one vector load per lane (its P consecutive channels) where kv_new allows it
  const int p = s.head_dim / vl;
  a.vec = p >= 4 && reinterpret_cast<uintptr_t>(kv_new) % (2 * p) == 0;
  for (int k = 0; k < 5; ++k) a.vec = a.vec && (strides[k] % p == 0);
  const int64_t warps = (vectors * vl + 31) / 32;
  const int64_t blocks = (warps + 3) / 4;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (s.head_dim == 128) {
    if (vl == 32)
      encode_kernel<128, 32><<<unsigned(blocks), 128, 0, stream>>>(a);
    else
      encode_kernel<128, 16><<<unsigned(blocks), 128, 0, stream>>>(a);
  } else {
    encode_kernel<64, 16><<<unsigned(blocks), 128, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace rq
