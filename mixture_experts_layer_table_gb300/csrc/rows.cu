// Row movement kernels: the pull dispatch (gather into expert-contiguous rows) and the
// fixed-order weighted merge (combine), plus the backward's reverse transfers.
//
// Pull dispatch: the expert side reads the token rows it needs and lays them out per
// expert itself ("把 MoE 通信延迟从 103μs 压到 18μs：Cursor 开源 GPU 内核 MoK",
// aientropygate.com, §03 ①); on one GPU the pull is a gather from HBM.  The combine ends in
// the weighted merge (same page, §04); each token's k rows are summed in the fixed order
// j = 0..k-1 in fp32, so the result is bitwise reproducible (no atomics).
#include <cuda_bf16.h>

#include "kernels.cuh"

namespace mok {

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// dst[r] = src[src_of[r] / k] for r < R; rows of H bf16 (H*2 bytes, a multiple of 16).
// One warp per row, 16-byte vectors, 4 independent loads in flight per lane.
__global__ void __launch_bounds__(256) gather_rows_kernel(const __nv_bfloat16* __restrict__ src,
                                                          const int32_t* __restrict__ src_of, int k, int R,
                                                          int vec_per_row, __nv_bfloat16* __restrict__ dst) {
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int r = blockIdx.x * warps + (threadIdx.x >> 5); r < R; r += gridDim.x * warps) {
    const int tok = src_of[r] / k;
    const uint4* s = reinterpret_cast<const uint4*>(src) + (size_t)tok * vec_per_row;
    uint4* d = reinterpret_cast<uint4*>(dst) + (size_t)r * vec_per_row;
    int i = lane;
    for (; i + 96 < vec_per_row; i += 128) {
      const uint4 a = ld_nc_v4(s + i), b = ld_nc_v4(s + i + 32), c = ld_nc_v4(s + i + 64),
                  e = ld_nc_v4(s + i + 96);
      st_v4_stream(d + i, a);
      st_v4_stream(d + i + 32, b);
      st_v4_stream(d + i + 64, c);
      st_v4_stream(d + i + 96, e);
    }
    for (; i < vec_per_row; i += 32) st_v4_stream(d + i, ld_nc_v4(s + i));
  }
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

// y[t] = sum_{j=0..k-1} w[t][j] * rows[row_of[t*k+j]]  (+ sum over the router support of
// dl[t][e] * w_router[e] when dl != nullptr), fp32 in the fixed order, rounded to bf16 once.
// rows are fp32 (expert outputs o, or per-row input gradients dX_g).
// `w` null means weight 1 (the backward's reverse dispatch of dX rows).
// Router support: the k selected experts (sparse) or all E experts (dense).
// One warp per token; each lane handles 8-column chunks (vec_per_row = H / 8).
template <int KMAX>
__global__ void __launch_bounds__(256)
    combine_kernel(const float* __restrict__ rows, const float* __restrict__ w,
                   const int32_t* __restrict__ row_of, int T, int k, int vec_per_row,
                   const float* __restrict__ dl, const __nv_bfloat16* __restrict__ w_router,
                   const int32_t* __restrict__ topk_idx, int E, int dense_router,
                   __nv_bfloat16* __restrict__ out) {
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += gridDim.x * warps) {
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
          va[j] = ld_nc_v4(p);
          vb[j] = ld_nc_v4(p + 1);
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
}

cudaError_t launch_gather_rows(const void* src, const int32_t* src_of, int k, int R, int H, void* dst,
                               int n_sm, cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  const int vec = H / 8;
  const int warps = 8;
  int blocks = (R + warps - 1) / warps;
  blocks = min(blocks, n_sm * 8);
  gather_rows_kernel<<<blocks, warps * 32, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), src_of, k, R,
                                                    vec, reinterpret_cast<__nv_bfloat16*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* rows, const float* w, const int32_t* row_of, int T, int k, int H,
                           const float* dl, const void* w_router, const int32_t* topk_idx, int E,
                           int dense_router, void* out, int n_sm, cudaStream_t st) {
  const int vec = H / 8;
  const int warps = 8;
  int blocks = (T + warps - 1) / warps;
  blocks = min(blocks, n_sm * 8);
  const float* r = rows;
  auto wr = reinterpret_cast<const __nv_bfloat16*>(w_router);
  auto o = reinterpret_cast<__nv_bfloat16*>(out);
  if (k <= 2)
    combine_kernel<2><<<blocks, warps * 32, 0, st>>>(r, w, row_of, T, k, vec, dl, wr, topk_idx, E, dense_router, o);
  else if (k <= 4)
    combine_kernel<4><<<blocks, warps * 32, 0, st>>>(r, w, row_of, T, k, vec, dl, wr, topk_idx, E, dense_router, o);
  else if (k <= 8)
    combine_kernel<8><<<blocks, warps * 32, 0, st>>>(r, w, row_of, T, k, vec, dl, wr, topk_idx, E, dense_router, o);
  else
    combine_kernel<16><<<blocks, warps * 32, 0, st>>>(r, w, row_of, T, k, vec, dl, wr, topk_idx, E, dense_router, o);
  return cudaGetLastError();
}

}  // namespace mok
