// The weighted merge of one token ("把 MoE 通信延迟从 103μs 压到 18μs：Cursor 开源 GPU 内核 MoK",
// aientropygate.com, §04: the measured layer ends with it): y[t] = sum_{j=0..k-1} w[t][j] *
// rows[row_of[t*k+j]], fp32 in the fixed order j = 0..k-1, rounded to bf16 once, so the result is
// bitwise reproducible; plus, for the backward's reverse dispatch, the router term
// sum_e dl[t][e] * w_router[e].  One warp per token, each lane 8 columns at a time.  Shared by the
// combine kernels (rows.cu) and the persistent ring forward (gemm_narrow.cuh), so both give the
// same bits.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

namespace mok {

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte load cached in L2 only: for rows written earlier in the same launch by other CTAs
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], uint4 v, float w) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = __bfloat1622float2(b[j]);
    acc[2 * j] = fmaf(w, f.x, acc[2 * j]);
    acc[2 * j + 1] = fmaf(w, f.y, acc[2 * j + 1]);
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
  uint4 o;
  uint32_t* p = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    p[j] = *reinterpret_cast<uint32_t*>(&b);
  }
  return o;
}

__device__ __forceinline__ void acc_f32x8(float (&acc)[8], uint4 a, uint4 b, float w) {
  acc[0] = fmaf(w, __uint_as_float(a.x), acc[0]);
  acc[1] = fmaf(w, __uint_as_float(a.y), acc[1]);
  acc[2] = fmaf(w, __uint_as_float(a.z), acc[2]);
  acc[3] = fmaf(w, __uint_as_float(a.w), acc[3]);
  acc[4] = fmaf(w, __uint_as_float(b.x), acc[4]);
  acc[5] = fmaf(w, __uint_as_float(b.y), acc[5]);
  acc[6] = fmaf(w, __uint_as_float(b.z), acc[6]);
  acc[7] = fmaf(w, __uint_as_float(b.w), acc[7]);
}

// Token t by one warp: rows fp32 (expert outputs o, or per-row input gradients dX_g); `w` null
// means weight 1 (the reverse dispatch of dX rows); `dl` null: no router term.  NC: the rows were
// written by an earlier launch (read through the non-coherent path); else by this launch (L2).
template <int KMAX, bool NC>
__device__ __forceinline__ void combine_token(const float* __restrict__ rows, const float* __restrict__ w,
                                              const int32_t* __restrict__ row_of, int t, int k, int vec_per_row,
                                              const float* __restrict__ dl,
                                              const __nv_bfloat16* __restrict__ w_router,
                                              const int32_t* __restrict__ topk_idx, int E, int dense_router,
                                              __nv_bfloat16* __restrict__ out, int lane) {
  int rj[KMAX];
  float wj[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (j < k) {
      rj[j] = row_of[(size_t)t * k + j];
      wj[j] = w ? w[(size_t)t * k + j] : 1.0f;
    }
  }
  for (int i = lane; i < vec_per_row; i += 32) {
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
    uint4 va[KMAX], vb[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) {
        const uint4* p = reinterpret_cast<const uint4*>(rows) + ((size_t)rj[j] * vec_per_row + i) * 2;
        va[j] = NC ? ld_nc_v4(p) : ld_cg_v4(p);
        vb[j] = NC ? ld_nc_v4(p + 1) : ld_cg_v4(p + 1);
      }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) acc_f32x8(acc, va[j], vb[j], wj[j]);
    if (dl != nullptr) {
      const int n_sup = dense_router ? E : k;
      for (int s = 0; s < n_sup; ++s) {
        const int e = dense_router ? s : topk_idx[(size_t)t * k + s];
        const float c = dl[(size_t)t * E + e];
        acc_bf16x8(acc, *(reinterpret_cast<const uint4*>(w_router) + (size_t)e * vec_per_row + i), c);
      }
    }
    reinterpret_cast<uint4*>(out)[(size_t)t * vec_per_row + i] = pack_bf16x8(acc);
  }
}

}  // namespace mok
