// MXFP8 helpers: E4M3 elements with one E8M0 scale per 32 consecutive elements (OCP
// Microscaling v1.0): shared exponent X = floor(log2(amax)) - 8, clamped to [-127, 127]
// (amax = 0 gives -127); elements are v * 2^-X rounded to nearest even into E4M3,
// saturating at +-448.  E8M0 stores X + 127.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace mok {

// Shared exponent of a block from its largest magnitude (an fp32 value, exact decision).
__device__ __forceinline__ int mx_exponent(float amax) {
  const uint32_t bits = __float_as_uint(amax) & 0x7fffffffu;
  const int ef = (int)(bits >> 23);
  if (ef == 0) return -127;  // zero or subnormal amax: floor(log2) - 8 is below -127
  return max(ef - 127 - 8, -127);
}

// 2^e as an fp32 value, e in [-149, 127] (subnormal results included).
__device__ __forceinline__ float exp2_int(int e) {
  if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

// Two fp32 values -> two E4M3 bytes (RNE, saturating): byte 0 = lo, byte 1 = hi.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two E4M3 bytes (byte 0 = lo element) -> two fp32 values (exact).
__device__ __forceinline__ float2 f32x2_from_e4m3x2(uint16_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

// Quantises 32 fp32 values in place to the MX grid (values become e4m3 * 2^X, exactly
// representable in bf16) and returns X.  `q` receives the 32 E4M3 bytes when non-null.
__device__ __forceinline__ int mx_quantize32(float (&v)[32], uint8_t* q) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const int X = mx_exponent(amax);
  const float inv = exp2_int(-X);  // -X in [-127, 127]: a normal number
  const float sc = exp2_int(X);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const uint16_t b = e4m3x2_from_f32(v[j] * inv, v[j + 1] * inv);
    if (q != nullptr) {
      q[j] = (uint8_t)(b & 0xff);
      q[j + 1] = (uint8_t)(b >> 8);
    }
    const float2 f = f32x2_from_e4m3x2(b);
    v[j] = f.x * sc;
    v[j + 1] = f.y * sc;
  }
  return X;
}

// The same quantisation with each 32-element block spread over 4 adjacent lanes of a warp (lane
// 4m + q holds elements 8q .. 8q+7 of block m): the block maximum is combined with two
// butterfly shuffles (a max is exact in any order), so the values are those of mx_quantize32.
// All 32 lanes of the warp must call it.
__device__ __forceinline__ void mx_quantize8_x4(float (&v)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int X = mx_exponent(amax);
  const float inv = exp2_int(-X);
  const float sc = exp2_int(X);
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float2 f = f32x2_from_e4m3x2(e4m3x2_from_f32(v[j] * inv, v[j + 1] * inv));
    v[j] = f.x * sc;
    v[j + 1] = f.y * sc;
  }
}

// mx_quantize8_x4 returning the E4M3 bytes (byte j = element j of this lane's 8, little-endian
// in `bytes`) and the block's exponent X instead of the dequantised values.  All 32 lanes of the
// warp must call it.
__device__ __forceinline__ int mx_quantize8_x4_e4m3(const float (&v)[8], uint2& bytes) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int X = mx_exponent(amax);
  const float inv = exp2_int(-X);
  uint32_t w[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t lo = e4m3x2_from_f32(v[4 * h] * inv, v[4 * h + 1] * inv);
    const uint32_t hi = e4m3x2_from_f32(v[4 * h + 2] * inv, v[4 * h + 3] * inv);
    w[h] = lo | (hi << 16);
  }
  bytes = make_uint2(w[0], w[1]);
  return X;
}

}  // namespace mok
