// mx.cuh -- MXFP8 (E4M3 elements, one UE8M0 scale per 32 elements) helpers
// shared by the quantising gather, the weight quantiser and the GEMM1
// epilogue.  Block format read as OCP MX (the pages name "MXFP8" only:
// leiphone "MoK..." section 02, MXFP8 paragraph).
//
// Scale-factor tiles: the scales of a 128-row x 128-element block (128 rows,
// 4 scale columns) are stored as one 512-byte tile; the scale of row r and
// 32-element block kb sits at byte 16*(r % 32) + 4*((r % 128) / 32) + (kb % 4).
// This is the order tcgen05.cp (32x128b, warpx4) needs to place row r's
// scales in TMEM lane r for tcgen05.mma kind::mxf8f6f4.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ int mx_sf_byte(int r, int kb) {
  return 16 * (r & 31) + 4 * ((r & 127) >> 5) + (kb & 3);
}

// Byte offset of the scale of (row r, 32-block kb) in a [rows, K] operand.
__device__ __forceinline__ size_t mx_sf_offset(size_t r, int kb, int k_groups) {
  return ((r >> 7) * (size_t)k_groups + (size_t)(kb >> 2)) * 512u + (size_t)mx_sf_byte((int)(r & 127), kb);
}

// UE8M0 exponent for a block with max |v| = amax: the smallest s with
// amax <= 448 * 2^s, clamped to [-127, 127]; amax = 0 or fp32-subnormal -> -127.
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int eb = (int)((b >> 23) & 0xFF);
  if (eb == 0) return -127;
  const uint32_t mant = b & 0x7FFFFFu;
  // amax = m * 2^q with m in [0.5, 1): q = eb - 126; m <= 0.875 <=> mant <= 0x600000
  const int s = (eb - 126) - ((mant <= 0x600000u) ? 9 : 8);
  return max(-127, min(127, s));
}

__device__ __forceinline__ float mx_exp2i(int s) {  // 2^s, |s| <= 126, exact
  return __uint_as_float((uint32_t)(s + 127) << 23);
}

__device__ __forceinline__ uint32_t mx_pack4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Quantise 32 fp32 values: writes 32 E4M3 codes (two uint4) and returns the
// scale byte (s + 127).  v * 2^-s is formed in two exact power-of-two steps.
__device__ __forceinline__ uint8_t mx_quant32(const float* v, uint4& lo, uint4& hi) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int s = mx_scale_exp(amax);
  const int s1 = -s / 2, s2 = -s - s1;
  const float f1 = mx_exp2i(s1), f2 = mx_exp2i(s2);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = mx_pack4(v[4 * i] * f1 * f2, v[4 * i + 1] * f1 * f2, v[4 * i + 2] * f1 * f2,
                    v[4 * i + 3] * f1 * f2);
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
  return (uint8_t)(s + 127);
}

// Quantise one value per lane of a warp whose 32 lanes form one block (a
// column of 32 rows): the block's scale from the warp-wide maximum, each
// lane's E4M3 code (same rounding and scale steps as mx_quant32).  Returns
// the code; *scale gets the scale byte (s + 127) in every lane.
__device__ __forceinline__ uint8_t mx_quant_lane(float v, uint8_t* scale) {
  // the bit patterns of non-negative floats order as their values: one
  // warp-wide integer max gives the block maximum of |v|
  const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
  const int s = mx_scale_exp(amax);
  const int s1 = -s / 2, s2 = -s - s1;
  const float y = v * mx_exp2i(s1) * mx_exp2i(s2);
  *scale = (uint8_t)(s + 127);
  return (uint8_t)(__nv_cvt_float2_to_fp8x2(make_float2(y, 0.f), __NV_SATFINITE, __NV_E4M3) & 0xFFu);
}

}  // namespace moe
