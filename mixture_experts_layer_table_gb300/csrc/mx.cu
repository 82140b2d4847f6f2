// MXFP8 preparation kernels: weight quantisation (E4M3 + E8M0 per 32 along K) and the
// dispatch gather with activation quantisation fused in ("把 MoE 通信延迟从 103μs 压到 18μs：
// Cursor 开源 GPU 内核 MoK", aientropygate.com, §03 ③: the MXFP8 activation quantisation sits
// on the dispatch / grouped GEMM / SwiGLU path instead of in a separate kernel).
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "mx.cuh"

namespace mok {

// w [E][N][K] bf16 -> q [E][N][K] E4M3 bytes, s [E][K/32][N] E8M0 bytes.  One thread per
// (e, k-block, n), n fastest so the scale stores are coalesced.
__global__ void __launch_bounds__(256)
    quantize_weights_kernel(const __nv_bfloat16* __restrict__ w, uint8_t* __restrict__ q, uint8_t* __restrict__ s,
                            int E, int N, int K) {
  const int KB = K / 32;
  const long long total = (long long)E * KB * N;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(i % N);
    const long long rest = i / N;
    const int kb = (int)(rest % KB);
    const int e = (int)(rest / KB);
    const size_t base = ((size_t)e * N + n) * K + (size_t)kb * 32;
    const uint4* src = reinterpret_cast<const uint4*>(w + base);
    float v[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 u = src[c];
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(b[j]);
        v[c * 8 + 2 * j] = f.x;
        v[c * 8 + 2 * j + 1] = f.y;
      }
    }
    __align__(16) uint8_t bytes[32];
    const int X = mx_quantize32(v, bytes);
    uint4* dst = reinterpret_cast<uint4*>(q + base);
    dst[0] = *reinterpret_cast<uint4*>(bytes);
    dst[1] = *reinterpret_cast<uint4*>(bytes + 16);
    s[((size_t)e * KB + kb) * N + n] = (uint8_t)(X + 127);
  }
}

// x_g[r] = MX(x[src_of[r] / k]) along H: each 32-element block quantised and stored back as
// bf16 (E4M3 * 2^X is exact in bf16).  One warp per row, one lane per 32-element block.
__global__ void __launch_bounds__(256)
    gather_rows_mx_kernel(const __nv_bfloat16* __restrict__ src, const int32_t* __restrict__ src_of, int k, int R,
                          int H, __nv_bfloat16* __restrict__ dst) {
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nb = H / 32;
  for (int r = blockIdx.x * warps + (threadIdx.x >> 5); r < R; r += gridDim.x * warps) {
    const int tok = src_of[r] / k;
    const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)tok * H);
    uint4* d = reinterpret_cast<uint4*>(dst + (size_t)r * H);
    for (int b = lane; b < nb; b += 32) {
      float v[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 u = s[b * 4 + c];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(h[j]);
          v[c * 8 + 2 * j] = f.x;
          v[c * 8 + 2 * j + 1] = f.y;
        }
      }
      mx_quantize32(v, nullptr);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 u;
        uint32_t* p = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          __nv_bfloat162 bb = __floats2bfloat162_rn(v[c * 8 + 2 * j], v[c * 8 + 2 * j + 1]);
          p[j] = *reinterpret_cast<uint32_t*>(&bb);
        }
        d[b * 4 + c] = u;
      }
    }
  }
}

cudaError_t launch_quantize_weights(const void* w, void* q, void* s, int E, int N, int K, int n_sm,
                                    cudaStream_t st) {
  const long long total = (long long)E * (K / 32) * N;
  long long blocks = (total + 255) / 256;
  if (blocks > (long long)n_sm * 64) blocks = (long long)n_sm * 64;
  quantize_weights_kernel<<<(int)blocks, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(w),
                                                       reinterpret_cast<uint8_t*>(q), reinterpret_cast<uint8_t*>(s),
                                                       E, N, K);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_mx(const void* src, const int32_t* src_of, int k, int R, int H, void* dst, int n_sm,
                                  cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  const int warps = 8;
  int blocks = (R + warps - 1) / warps;
  blocks = min(blocks, n_sm * 8);
  gather_rows_mx_kernel<<<blocks, warps * 32, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), src_of, k, R, H,
                                                       reinterpret_cast<__nv_bfloat16*>(dst));
  return cudaGetLastError();
}

}  // namespace mok
