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

// Four E4M3 bytes w (byte i = element i) times 2^X -> four bf16 values as two bf16x2 words
// (lo = elements 0, 1; hi = elements 2, 3), with integer operations only: the sign, 4 exponent
// and 3 mantissa bits of each byte are moved to the bf16 positions and (120 + X) is added to
// the exponent (E4M3 bias 7 -> bf16 bias 127).  Valid when no byte has a zero exponent field
// (zero or subnormal) and -120 <= X <= 119; returns false otherwise (the caller converts the
// slow way).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(a), "r"(sel));
  return d;
}

// Nonzero when some byte of w has a zero exponent field (an E4M3 zero or subnormal).
__device__ __forceinline__ uint32_t e4m3_zero_exponent_bytes(uint32_t w) {
  const uint32_t t = w & 0x78787878u;
  return (t - 0x01010101u) & ~t & 0x80808080u;
}

// Four E4M3 bytes with nonzero exponents, times 2^X for -120 <= X <= 119.  prmt with the
// sign-replicate selector bit builds [sign(b1)][b1][sign(b0)][b0]; shifted left by 4 this puts
// each byte's exponent and mantissa at bf16 bits 10..4 and its sign at bit 15 of its half,
// the mask drops the rest, and adding (120 + X) << 7 rebiases the exponent.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t bias2, uint32_t& lo, uint32_t& hi) {
  lo = ((prmt(w, 0x9180u) << 4) & 0x87F087F0u) + bias2;
  hi = ((prmt(w, 0xB3A2u) << 4) & 0x87F087F0u) + bias2;
}

// Slow path for a 16-byte chunk that holds a zero / subnormal or has an extreme scale (kept
// out of line so that the common path is a real branch, not a predicated copy of this one): the
// 16 values, times 2^X, as bf16 into dst0 (elements 0-7) and dst1 (elements 8-15).  It stores
// them itself so that the common path keeps its values in registers.
static __device__ __noinline__ void e4m3x16_to_bf16x16_slow(uint4 raw, int X, uint4* dst0, uint4* dst1) {
  const float sc = exp2_int(X);
  const uint16_t* pairs = reinterpret_cast<const uint16_t*>(&raw);
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 f = f32x2_from_e4m3x2(pairs[j]);
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x * sc, f.y * sc);
    o[j] = *reinterpret_cast<uint32_t*>(&b);
  }
  *dst0 = make_uint4(o[0], o[1], o[2], o[3]);
  *dst1 = make_uint4(o[4], o[5], o[6], o[7]);
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
