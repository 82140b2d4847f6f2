// MXFP8 preparation kernels: weight quantisation (E4M3 + E8M0 per 32 along K) and the
// dispatch gather with activation quantisation fused in ("把 MoE 通信延迟从 103μs 压到 18μs：
// Cursor 开源 GPU 内核 MoK", aientropygate.com, §03 ③: the MXFP8 activation quantisation sits
// on the dispatch / grouped GEMM / SwiGLU path instead of in a separate kernel).
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.cuh"
#include "mx.cuh"
#include "mx_tiles.h"
#include "ptx.cuh"

namespace mok {

// w [E][N][K] bf16 -> q [E][N][K] E4M3 bytes, s [E][N/128][K/128][512] E8M0 bytes: one 512-byte
// block per 128-row tile and 128-element K stage, in the order tcgen05.cp puts it into TMEM
// (mx_tiles.h).  With gate_up_I > 0 (W13, N = 2I) tile t holds the gate rows 64 t .. 64 t + 63 and
// the up rows I + 64 t .. I + 64 t + 63 (the rows one CTA of the SwiGLU GEMM multiplies).  One
// thread per (e, k-block, n), n fastest.
__global__ void __launch_bounds__(256)
    quantize_weights_kernel(const __nv_bfloat16* __restrict__ w, uint8_t* __restrict__ q, uint8_t* __restrict__ s,
                            int E, int N, int K, int gate_up_I) {
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
    int tile = n >> 7, local = n & 127;
    if (gate_up_I > 0) {
      const int half = n / gate_up_I, ii = n - half * gate_up_I;
      tile = ii >> 6;
      local = half * 64 + (ii & 63);
    }
    s[(((size_t)e * (N / 128) + tile) * (K / 128) + kb / 4) * MX_SF_BLOCK + mx_sf_byte(local, kb & 3)] =
        (uint8_t)(X + 127);
  }
}

// x_g[r] = MX(x[src_of[r] / k]) along H: each 32-element block quantised and stored back as
// bf16 (E4M3 * 2^X is exact in bf16).  One short-lived block of 128 threads per destination row
// (as the bf16 gather): 16-byte coalesced loads and stores, 4 adjacent lanes per 32-element block
// (mx_quantize8_x4), the source rows marked L2 evict-last (each is read k times).  A persistent
// version with one lane per 32-element block (64-byte strided accesses) moved 3.6 TB/s.
constexpr int GATHER_MX_THREADS = 128;
__global__ void __launch_bounds__(GATHER_MX_THREADS)
    gather_rows_mx_kernel(const __nv_bfloat16* __restrict__ src, const int32_t* __restrict__ src_of, int k,
                          int vec_per_row, __nv_bfloat16* __restrict__ dst) {
  constexpr int V = 8;
  const int r = blockIdx.x;
  const int tok = src_of[r] / k;
  const uint64_t keep = l2_policy_evict_last();
  const uint4* s = reinterpret_cast<const uint4*>(src) + (size_t)tok * vec_per_row;
  uint4* d = reinterpret_cast<uint4*>(dst) + (size_t)r * vec_per_row;
  for (int base = threadIdx.x; base < vec_per_row; base += GATHER_MX_THREADS * V) {
    uint4 u[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int i = base + j * GATHER_MX_THREADS;  // a warp's 32 lanes are all in range or none
      if (i < vec_per_row)
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                     : "=r"(u[j].x), "=r"(u[j].y), "=r"(u[j].z), "=r"(u[j].w)
                     : "l"(s + i), "l"(keep));
    }
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int i = base + j * GATHER_MX_THREADS;
      if (i < vec_per_row) {
        float v[8];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[j]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(h[q]);
          v[2 * q] = f.x;
          v[2 * q + 1] = f.y;
        }
        mx_quantize8_x4(v);
        uint4 o;
        uint32_t* p = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          __nv_bfloat162 bb = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
          p[q] = *reinterpret_cast<uint32_t*>(&bb);
        }
        asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(d + i), "r"(o.x), "r"(o.y), "r"(o.z),
                     "r"(o.w)
                     : "memory");
      }
    }
  }
}

// Backward-direction MXFP8 weights: w [E][N][K] bf16 -> wt [E][K][N] E4M3, each row of wt (a column
// of w) quantised in 32-element blocks along N, scales s [E][K/128][N/128][512] (the layout of
// quantize_weights_kernel for the transposed matrix).  One thread per (e, k, 32-block of N), k
// fastest: a warp reads 32 consecutive k of each of its 32 rows (64-byte segments) and writes 32
// bytes of its own row of wt.
__global__ void __launch_bounds__(256)
    quantize_transpose_kernel(const __nv_bfloat16* __restrict__ w, uint8_t* __restrict__ wt, uint8_t* __restrict__ s,
                              int E, int N, int K) {
  const int NB = N / 32;
  const long long total = (long long)E * NB * K;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(idx % K);
    const long long rest = idx / K;
    const int nb = (int)(rest % NB);
    const int e = (int)(rest / NB);
    const __nv_bfloat16* src = w + ((size_t)e * N + (size_t)nb * 32) * K + k;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __bfloat162float(src[(size_t)j * K]);
    __align__(16) uint8_t bytes[32];
    const int X = mx_quantize32(v, bytes);
    uint4* dst = reinterpret_cast<uint4*>(wt + ((size_t)e * K + k) * N + (size_t)nb * 32);
    dst[0] = *reinterpret_cast<uint4*>(bytes);
    dst[1] = *reinterpret_cast<uint4*>(bytes + 16);
    s[(((size_t)e * (K / 128) + k / 128) * (N / 128) + nb / 4) * MX_SF_BLOCK + mx_sf_byte(k & 127, nb & 3)] =
        (uint8_t)(X + 127);
  }
}

// The dispatch of the MXFP8 forward on the FP8 tensor path: x_q[p] = E4M3 bytes of
// x[src_of[r] / k] along H, at padded row p = 32 blk_off[e] + (r - offsets[e]) of the row's expert
// e, and the row's scales into the four row-group blocks that hold them (mx_tiles.h).  Blocks
// [0, R) are rows, as gather_rows_mx_kernel: 128 threads, 16-byte loads, 4 adjacent lanes per
// 32-element block (mx_quantize8_x4_e4m3), one 8-byte store per lane.  Block R + e zero-fills the
// padding rows of expert e (their bytes and scales), so that the GEMM reads zeros there.
__global__ void __launch_bounds__(GATHER_MX_THREADS)
    gather_rows_mxf8_kernel(const __nv_bfloat16* __restrict__ src, const int32_t* __restrict__ src_of,
                            const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ offsets,
                            const int32_t* __restrict__ blk_off, int k, int R, int H, uint8_t* __restrict__ xq,
                            uint8_t* __restrict__ xsf) {
  constexpr int V = 8;
  const int vec_per_row = H / 8;
  const int S = H / MX_BK;
  if ((int)blockIdx.x < R) {
    const int r = blockIdx.x;
    const int a = src_of[r];
    const int tok = a / k;
    const int e = topk_idx[a];
    const int p = MX_ROW_ALIGN * blk_off[e] + (r - offsets[e]);
    const uint64_t keep = l2_policy_evict_last();
    const uint4* s = reinterpret_cast<const uint4*>(src) + (size_t)tok * vec_per_row;
    uint2* d = reinterpret_cast<uint2*>(xq + (size_t)p * H);
    // H a multiple of 128: a warp's 32 lanes (256 elements) may reach past the row by 16 lanes;
    // those lanes quantise zeros alongside (the 4-lane shuffles of a block see every lane) and
    // store nothing.  Blocks (4 lanes) are whole: in the row or past it.
    const int lane = threadIdx.x & 31;
    for (int base = threadIdx.x; base - lane < vec_per_row; base += GATHER_MX_THREADS * V) {
      uint4 u[V];
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int i = base + j * GATHER_MX_THREADS;
        u[j] = make_uint4(0u, 0u, 0u, 0u);
        if (i < vec_per_row)
          asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                       : "=r"(u[j].x), "=r"(u[j].y), "=r"(u[j].z), "=r"(u[j].w)
                       : "l"(s + i), "l"(keep));
      }
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int i = base + j * GATHER_MX_THREADS;
        if (base - lane + j * GATHER_MX_THREADS < vec_per_row) {  // the warp's first lane is in the row
          float v[8];
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[j]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(h[q]);
            v[2 * q] = f.x;
            v[2 * q + 1] = f.y;
          }
          uint2 bytes;
          const int X = mx_quantize8_x4_e4m3(v, bytes);
          if (i < vec_per_row) d[i] = bytes;
          if (i < vec_per_row && (i & 3) == 0) {  // the first lane of the block stores its scale
            const int kb = i >> 2;
            const int g_top = p >> 5;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int g = g_top - jj;
              if (g >= 0)
                xsf[((size_t)g * S + (kb >> 2)) * MX_SF_BLOCK + (p & 31) * 16 + jj * 4 + (kb & 3)] = (uint8_t)(X + 127);
            }
          }
        }
      }
    }
  } else {
    const int e = (int)blockIdx.x - R;
    const int p_end = MX_ROW_ALIGN * blk_off[e + 1];
    for (int p = MX_ROW_ALIGN * blk_off[e] + (offsets[e + 1] - offsets[e]); p < p_end; ++p) {
      uint2* d = reinterpret_cast<uint2*>(xq + (size_t)p * H);
      for (int i = threadIdx.x; i < vec_per_row; i += GATHER_MX_THREADS) d[i] = make_uint2(0u, 0u);
      const int g_top = p >> 5;
      for (int kb = threadIdx.x; kb < H / 32; kb += GATHER_MX_THREADS) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int g = g_top - jj;
          if (g >= 0) xsf[((size_t)g * S + (kb >> 2)) * MX_SF_BLOCK + (p & 31) * 16 + jj * 4 + (kb & 3)] = 0;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- MXFP8 backward operands
// In the backward every GEMM operand is quantised along that GEMM's reduction dimension: for
// the weight gradients that is the row (token) axis inside each expert's segment, in blocks of 32
// rows that start at the segment's first row (a ragged last block is padded with zeros), for the
// transposed weights the row axis of W2[e] (H) and W13[e] (2I).  Quantised values are stored as
// their exact bf16 values.

// blk_off[e] = number of 32-row blocks of the segments before e (blk_off[E] = total).
__global__ void __launch_bounds__(1024) mx_block_offsets_kernel(const int32_t* __restrict__ offsets, int E,
                                                                 int32_t* __restrict__ blk_off) {
  __shared__ int32_t sc[1024];
  const int t = threadIdx.x;
  sc[t] = t < E ? (offsets[t + 1] - offsets[t] + 31) / 32 : 0;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {  // inclusive scan
    const int32_t v = t >= d ? sc[t - d] : 0;
    __syncthreads();
    sc[t] += v;
    __syncthreads();
  }
  if (t < E) blk_off[t + 1] = sc[t];
  if (t == 0) blk_off[0] = 0;
}

enum MxRowSrc { MXR_PLAIN = 0, MXR_SPLIT = 1, MXR_SWIGLU = 2, MXR_GATHER = 3, MXR_GATHER_GATE = 4 };

struct MxRowsArgs {
  int C;                          // columns (output row length)
  int E;
  int seg_len;                    // > 0: E segments of seg_len rows; 0: segments from offsets
  const int32_t* offsets;         // [E+1]
  const int32_t* blk_off;         // [E+1] from mx_block_offsets_kernel
  const __nv_bfloat16* in0;       // PLAIN / SPLIT hi [rows][C]; GATHER*: token rows [T][C]
  const __nv_bfloat16* in1;       // SPLIT lo
  const float* hu;                // SWIGLU: h | u [rows][2C]
  const float* gate_row;          // GATHER_GATE: gate of each row
  const int32_t* src_of;          // GATHER*: row -> assignment (token = src_of / k)
  int k;
  __nv_bfloat16* out;             // [rows][C]
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float* f) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 t = __bfloat1622float2(b[q]);
    f[2 * q] = t.x;
    f[2 * q + 1] = t.y;
  }
}

// Values of row r, columns c .. c+7 (c a multiple of 8), from the source.
template <int SRC>
__device__ __forceinline__ void mx_row_values8(const MxRowsArgs& a, int r, int c, float* f) {
  if (SRC == MXR_PLAIN || SRC == MXR_SPLIT) {
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.in0 + (size_t)r * a.C + c), f);
    if (SRC == MXR_SPLIT) {
      float l[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.in1 + (size_t)r * a.C + c), l);
#pragma unroll
      for (int q = 0; q < 8; ++q) f[q] += l[q];
    }
  } else if (SRC == MXR_SWIGLU) {
    const float4* hp = reinterpret_cast<const float4*>(a.hu + (size_t)r * 2 * a.C + c);
    const float4* up = reinterpret_cast<const float4*>(a.hu + (size_t)r * 2 * a.C + a.C + c);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float4 h4 = hp[q], u4 = up[q];
      const float hv[4] = {h4.x, h4.y, h4.z, h4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
      for (int z = 0; z < 4; ++z) f[4 * q + z] = hv[z] / (1.0f + __expf(-hv[z])) * uv[z];
    }
  } else {
    const int tok = a.src_of[r] / a.k;
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.in0 + (size_t)tok * a.C + c), f);
    if (SRC == MXR_GATHER_GATE) {
      const float g = a.gate_row[r];
#pragma unroll
      for (int q = 0; q < 8; ++q) f[q] *= g;
    }
  }
}

// One short-lived CTA per (32-row block, 256 columns): the 32 x 256 values are staged in shared
// memory with 16-byte loads along the rows, thread c quantises column c as one MX block, the
// quantised values go back into the tile and leave as 16-byte stores along the rows.  Staged rows
// are 260 floats apart (16-byte aligned; the column reads hit 32 different banks).  C is a
// multiple of 128: the last chunk of a row may hold 128 columns, the rest of its tile is zeros that
// are quantised and not stored.  (A persistent version that stored one bf16 per thread per row, with 8-way
// bank conflicts on the staging, ran the x_g and dY_g passes at 1.3 TB/s.)
constexpr int MXQ_LD = 260;
template <int SRC>
__global__ void __launch_bounds__(256) mx_quant_rows_kernel(const MxRowsArgs a) {
  __shared__ __align__(16) float tile[32 * MXQ_LD];
  const int nchunk = (a.C + 255) / 256;
  const int nblk = a.seg_len > 0 ? a.E * (a.seg_len / 32) : a.blk_off[a.E];
  const long long items = (long long)nblk * nchunk;
  const long long w = blockIdx.x;
  if (w >= items) return;  // the grid is an upper bound of the items
  const int b = (int)(w / nchunk);
  const int c0 = (int)(w - (long long)b * nchunk) * 256;
  const int cols = min(256, a.C - c0);
  int r0, nrows;
  if (a.seg_len > 0) {
    r0 = b * 32;
    nrows = 32;
  } else {
    int lo = 0, hi = a.E;  // largest e with blk_off[e] <= b (the last of equal starts owns blocks)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(&a.blk_off[mid]) <= b) lo = mid; else hi = mid;
    }
    r0 = __ldg(&a.offsets[lo]) + 32 * (b - __ldg(&a.blk_off[lo]));
    nrows = min(32, __ldg(&a.offsets[lo + 1]) - r0);
  }
  // stage: 32 rows x 32 chunks of 8 columns, 4 chunks per thread (a warp covers one row)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = threadIdx.x + 256 * i;
    const int row = idx >> 5, ch = idx & 31;
    float f[8];
    if (row < nrows && 8 * ch < cols) {
      mx_row_values8<SRC>(a, r0 + row, c0 + 8 * ch, f);
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) f[q] = 0.0f;  // the ragged last block is padded with zeros
    }
    float4* t4 = reinterpret_cast<float4*>(&tile[row * MXQ_LD + 8 * ch]);
    t4[0] = make_float4(f[0], f[1], f[2], f[3]);
    t4[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
  __syncthreads();
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = tile[j * MXQ_LD + threadIdx.x];
  mx_quantize32(v, nullptr);
  __syncthreads();  // every column has been read before the tile is overwritten
#pragma unroll
  for (int j = 0; j < 32; ++j) tile[j * MXQ_LD + threadIdx.x] = v[j];
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = threadIdx.x + 256 * i;
    const int row = idx >> 5, ch = idx & 31;
    if (row < nrows && 8 * ch < cols) {
      const float4* t4 = reinterpret_cast<const float4*>(&tile[row * MXQ_LD + 8 * ch]);
      const float4 x0 = t4[0], x1 = t4[1];
      uint4 o;
      uint32_t* p = reinterpret_cast<uint32_t*>(&o);
      __nv_bfloat162 b0 = __floats2bfloat162_rn(x0.x, x0.y), b1 = __floats2bfloat162_rn(x0.z, x0.w);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(x1.x, x1.y), b3 = __floats2bfloat162_rn(x1.z, x1.w);
      p[0] = *reinterpret_cast<uint32_t*>(&b0);
      p[1] = *reinterpret_cast<uint32_t*>(&b1);
      p[2] = *reinterpret_cast<uint32_t*>(&b2);
      p[3] = *reinterpret_cast<uint32_t*>(&b3);
      *reinterpret_cast<uint4*>(a.out + (size_t)(r0 + row) * a.C + c0 + 8 * ch) = o;
    }
  }
}

// out[r] = MX(hi[r] + lo[r]) along the row, blocks of 32 columns.  One thread per block.
__global__ void __launch_bounds__(256)
    mx_quant_cols_kernel(const __nv_bfloat16* __restrict__ hi, const __nv_bfloat16* __restrict__ lo, long long R,
                         int C, __nv_bfloat16* __restrict__ out) {
  const int nb = C / 32;
  const long long total = R * nb;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const size_t base = (size_t)i * 32;  // row-major: block i covers elements 32i .. 32i+31
    const uint4* h4 = reinterpret_cast<const uint4*>(hi + base);
    const uint4* l4 = reinterpret_cast<const uint4*>(lo + base);
    float v[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 uh = h4[c], ul = l4[c];
      const __nv_bfloat162* bh = reinterpret_cast<const __nv_bfloat162*>(&uh);
      const __nv_bfloat162* bl = reinterpret_cast<const __nv_bfloat162*>(&ul);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 fh = __bfloat1622float2(bh[j]), fl = __bfloat1622float2(bl[j]);
        v[c * 8 + 2 * j] = fh.x + fl.x;
        v[c * 8 + 2 * j + 1] = fh.y + fl.y;
      }
    }
    mx_quantize32(v, nullptr);
    uint4* d = reinterpret_cast<uint4*>(out + base);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 u;
      uint32_t* p = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 bb = __floats2bfloat162_rn(v[c * 8 + 2 * j], v[c * 8 + 2 * j + 1]);
        p[j] = *reinterpret_cast<uint32_t*>(&bb);
      }
      d[c] = u;
    }
  }
}

cudaError_t launch_mx_block_offsets(const int32_t* offsets, int E, int32_t* blk_off, cudaStream_t st) {
  if (E > 1024) return cudaErrorInvalidValue;
  mx_block_offsets_kernel<<<1, 1024, 0, st>>>(offsets, E, blk_off);
  return cudaGetLastError();
}

cudaError_t launch_mx_quant_rows(int src, int rows_bound, int C, int E, int seg_len, const int32_t* offsets,
                                 const int32_t* blk_off, const void* in0, const void* in1, const float* hu,
                                 const float* gate_row, const int32_t* src_of, int k, void* out, int n_sm,
                                 cudaStream_t st) {
  MxRowsArgs a;
  a.C = C;
  a.E = E;
  a.seg_len = seg_len;
  a.offsets = offsets;
  a.blk_off = blk_off;
  a.in0 = reinterpret_cast<const __nv_bfloat16*>(in0);
  a.in1 = reinterpret_cast<const __nv_bfloat16*>(in1);
  a.hu = hu;
  a.gate_row = gate_row;
  a.src_of = src_of;
  a.k = k;
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  if ((seg_len > 0 && seg_len % 32 != 0) || C % 128 != 0) return cudaErrorInvalidValue;
  // an upper bound of the work items sizes the grid; the kernel reads the exact count
  // an upper bound of the work items sizes the grid (one item per CTA); the kernel reads the
  // exact count
  (void)n_sm;
  const long long items = (long long)((rows_bound + 31) / 32 + E) * ((C + 255) / 256);
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int blocks = (int)std::max<long long>(items, 1);
  switch (src) {
    case MXR_PLAIN: mx_quant_rows_kernel<MXR_PLAIN><<<blocks, 256, 0, st>>>(a); break;
    case MXR_SPLIT: mx_quant_rows_kernel<MXR_SPLIT><<<blocks, 256, 0, st>>>(a); break;
    case MXR_SWIGLU: mx_quant_rows_kernel<MXR_SWIGLU><<<blocks, 256, 0, st>>>(a); break;
    case MXR_GATHER: mx_quant_rows_kernel<MXR_GATHER><<<blocks, 256, 0, st>>>(a); break;
    case MXR_GATHER_GATE: mx_quant_rows_kernel<MXR_GATHER_GATE><<<blocks, 256, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_mx_quant_cols(const void* hi, const void* lo, long long R, int C, void* out, int n_sm,
                                 cudaStream_t st) {
  if (C % 32 != 0) return cudaErrorInvalidValue;
  const long long total = R * (C / 32);
  if (total == 0) return cudaSuccess;
  const int blocks = (int)std::min<long long>((total + 255) / 256, (long long)n_sm * 16);
  mx_quant_cols_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(hi),
                                               reinterpret_cast<const __nv_bfloat16*>(lo), R, C,
                                               reinterpret_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_quantize_weights(const void* w, void* q, void* s, int E, int N, int K, int gate_up_I, int n_sm,
                                    cudaStream_t st) {
  const long long total = (long long)E * (K / 32) * N;
  long long blocks = (total + 255) / 256;
  if (blocks > (long long)n_sm * 64) blocks = (long long)n_sm * 64;
  quantize_weights_kernel<<<(int)blocks, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(w),
                                                       reinterpret_cast<uint8_t*>(q), reinterpret_cast<uint8_t*>(s),
                                                       E, N, K, gate_up_I);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_mx(const void* src, const int32_t* src_of, int k, int R, int H, void* dst, int n_sm,
                                  cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  (void)n_sm;
  gather_rows_mx_kernel<<<R, GATHER_MX_THREADS, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), src_of, k, H / 8,
                                                         reinterpret_cast<__nv_bfloat16*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_quantize_transpose(const void* w, void* wt_q, void* wt_s, int E, int N, int K, int n_sm,
                                      cudaStream_t st) {
  const long long total = (long long)E * (N / 32) * K;
  long long blocks = (total + 255) / 256;
  if (blocks > (long long)n_sm * 64) blocks = (long long)n_sm * 64;
  if (blocks <= 0) return cudaSuccess;
  quantize_transpose_kernel<<<(int)blocks, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(w),
                                                         reinterpret_cast<uint8_t*>(wt_q), reinterpret_cast<uint8_t*>(wt_s),
                                                         E, N, K);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_mxf8(const void* x, const int32_t* src_of, const int32_t* topk_idx,
                                    const int32_t* offsets, const int32_t* blk_off, int k, int R, int H, int E,
                                    void* xq, void* xsf, cudaStream_t st) {
  if (R + E == 0) return cudaSuccess;
  gather_rows_mxf8_kernel<<<R + E, GATHER_MX_THREADS, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), src_of, topk_idx, offsets, blk_off, k, R, H,
      reinterpret_cast<uint8_t*>(xq), reinterpret_cast<uint8_t*>(xsf));
  return cudaGetLastError();
}

}  // namespace mok
