// Row movement kernels: the pull dispatch (gather into expert-contiguous rows) and the
// fixed-order weighted merge (combine), plus the backward's reverse transfers.
//
// Pull dispatch: the expert side reads the token rows it needs and lays them out per
// expert itself ("把 MoE 通信延迟从 103μs 压到 18μs：Cursor 开源 GPU 内核 MoK",
// aientropygate.com, §03 ①); on one GPU the pull is a gather from HBM.  The combine ends in
// the weighted merge (same page, §04); each token's k rows are summed in the fixed order
// j = 0..k-1 in fp32, so the result is bitwise reproducible (no atomics).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "combine.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace mok {

// 16-byte load that asks L2 to keep the line (policy from createpolicy ... evict_last)
__device__ __forceinline__ uint4 ld_nc_v4_keep(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

__device__ __forceinline__ void st_v4_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// dst[r] = src[src_of[r] / k] for r < R; rows of H bf16 (H*2 bytes, a multiple of 16).
// One short-lived block of 128 threads per destination row: each thread loads its V 16-byte
// vectors of the row (all in flight at once), then stores them; blocks run in row order, so the
// rows being written at any time form one contiguous window of dst.  Measured on GB300: a
// persistent grid-stride version (one warp per row, 4 loads in flight per lane) wrote 3.9-4.7
// TB/s; a fill of short-lived 16 KB blocks reaches 7.8 TB/s where grid-stride loops reach 6.5.
constexpr int GATHER_THREADS = 128;
template <int V>
__global__ void __launch_bounds__(GATHER_THREADS) gather_rows_kernel(const __nv_bfloat16* __restrict__ src,
                                                                     const int32_t* __restrict__ src_of, int k,
                                                                     int vec_per_row,
                                                                     __nv_bfloat16* __restrict__ dst) {
  const int r = blockIdx.x;
  const int tok = src_of[r] / k;
  // each source row is read k times, by blocks far apart in time: keep it in L2
  const uint64_t keep = l2_policy_evict_last();
  const uint4* s = reinterpret_cast<const uint4*>(src) + (size_t)tok * vec_per_row;
  uint4* d = reinterpret_cast<uint4*>(dst) + (size_t)r * vec_per_row;
  for (int base = threadIdx.x; base < vec_per_row; base += GATHER_THREADS * V) {
    uint4 v[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int i = base + j * GATHER_THREADS;
      if (i < vec_per_row) v[j] = ld_nc_v4_keep(s + i, keep);
    }
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int i = base + j * GATHER_THREADS;
      if (i < vec_per_row) st_v4_stream(d + i, v[j]);
    }
  }
}

// Ring backward: block r replays dispatched row r unless the ring still holds it.  Every block
// reads the two stamps (L2-resident after the first) and decides the same way.
__global__ void __launch_bounds__(GATHER_THREADS)
    ring_replay_kernel(const __nv_bfloat16* __restrict__ src, const int32_t* __restrict__ src_of, int k,
                       int vec_per_row, __nv_bfloat16* __restrict__ dst, int head_rows,
                       const unsigned long long* __restrict__ ws_stamp, const unsigned long long* __restrict__ ctx_stamp,
                       unsigned long long ctx_addr) {
  const int r = blockIdx.x;
  const bool resident = ws_stamp[0] == ctx_addr && ws_stamp[1] == ctx_stamp[0];
  if (resident && r >= head_rows) return;
  const int tok = src_of[r] / k;
  const uint64_t keep = l2_policy_evict_last();
  const uint4* s = reinterpret_cast<const uint4*>(src) + (size_t)tok * vec_per_row;
  uint4* d = reinterpret_cast<uint4*>(dst) + (size_t)r * vec_per_row;
  for (int i = threadIdx.x; i < vec_per_row; i += GATHER_THREADS) st_v4_stream(d + i, ld_nc_v4_keep(s + i, keep));
}

__global__ void ring_stamp_kernel(unsigned long long* ctx_stamp, unsigned long long* ws_stamp,
                                  unsigned long long ctx_addr) {
  const unsigned long long n = ctx_stamp[0] + 1;
  ctx_stamp[0] = n;
  ws_stamp[0] = ctx_addr;
  ws_stamp[1] = n;
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
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += gridDim.x * warps)
    combine_token<KMAX, true>(rows, w, row_of, t, k, vec_per_row, dl, w_router, topk_idx, E, dense_router, out, lane);
}

cudaError_t launch_gather_rows(const void* src, const int32_t* src_of, int k, int R, int H, void* dst,
                               int n_sm, cudaStream_t st) {
  (void)n_sm;
  if (R == 0) return cudaSuccess;
  const int vec = H / 8;
  gather_rows_kernel<8><<<R, GATHER_THREADS, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), src_of, k, vec,
                                                      reinterpret_cast<__nv_bfloat16*>(dst));
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

// bf16 -> fp16, 8 elements per thread per step (16-byte loads and stores; a ragged tail element by
// element).  Round to nearest even: exact for bf16 values of magnitude 2^-14 .. 65504 (fp16 normals
// hold every 8-bit bf16 significand), smaller ones become fp16 subnormals (absolute error <= 2^-25).
__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const __nv_bfloat16* __restrict__ src,
                                                          __half* __restrict__ dst, long long n) {
  const long long n8 = n / 8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[i];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
    uint4 o;
    __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) h[q] = __float22half2_rn(__bfloat1622float2(b[q]));
    reinterpret_cast<uint4*>(dst)[i] = o;
  }
  for (long long i = n8 * 8 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = __float2half_rn(__bfloat162float(src[i]));
}

cudaError_t launch_bf16_to_f16(const void* src, void* dst, long long n, int n_sm, cudaStream_t st) {
  bf16_to_f16_kernel<<<n_sm * 8, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src),
                                               reinterpret_cast<__half*>(dst), n);
  return cudaGetLastError();
}

cudaError_t launch_ring_replay(const void* x, const int32_t* src_of, int k, int R, int H, void* x_rows, int head_rows,
                               const unsigned long long* ws_stamp, const unsigned long long* ctx_stamp,
                               unsigned long long ctx_addr, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  ring_replay_kernel<<<R, GATHER_THREADS, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(x), src_of, k, H / 8,
                                                   reinterpret_cast<__nv_bfloat16*>(x_rows), head_rows, ws_stamp,
                                                   ctx_stamp, ctx_addr);
  return cudaGetLastError();
}

cudaError_t launch_ring_stamp(unsigned long long* ctx_stamp, unsigned long long* ws_stamp, unsigned long long ctx_addr,
                              cudaStream_t st) {
  ring_stamp_kernel<<<1, 1, 0, st>>>(ctx_stamp, ws_stamp, ctx_addr);
  return cudaGetLastError();
}

}  // namespace mok
