// Router top-k, schedule table and router backward kernels.
//
// The schedule table is the "unified schedule table" of "Mixture-of-Kittens (MoK)"
// (sd114.wiki, pull-dispatch section): for the assignments a = t*k + j it counts the rows
// of each expert, takes the exclusive prefix sum, and gives every assignment its row in
// an expert-contiguous order (the three jobs listed in aientropygate.com §02).  It is a
// stable counting sort, so it is exact and reproducible.
#include <cuda_bf16.h>

#include "kernels.cuh"
#include "status.cuh"

namespace mok {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 16;

// ----------------------------------------------------------------------------- top-k
// One warp per token.  Scores: softmax over the E logits or elementwise sigmoid.
// Selection score = score + bias (bias nullable); the k best are taken best-first, ties
// to the lower expert index.  Gates = scores at the selected experts, renormalised over
// the k when requested, times route_scale.
// C: experts per lane (32 * C >= E), so that the scans run over the chunks that exist.
template <int C>
__global__ void topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                            const int32_t* __restrict__ given, int T, int E, int k, int router,
                            int renorm, float route_scale, int32_t* __restrict__ topk_idx,
                            float* __restrict__ gates, float* __restrict__ scores_out,
                            int* status) {
  static_assert(C >= 1 && 32 * C <= kMaxE, "experts per lane");
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float s[C];
  // logits == nullptr: the selection must be given; gates are then not produced
  const float* lrow = logits != nullptr ? logits + (size_t)t * E : nullptr;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int e = c * 32 + lane;
    s[c] = (e < E && logits != nullptr) ? lrow[e] : (e < E ? 0.0f : -INFINITY);
  }
  if (router == 0) {  // softmax, max-shifted
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < C; ++c) m = fmaxf(m, s[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.0f;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int e = c * 32 + lane;
      s[c] = (e < E) ? expf(s[c] - m) : 0.0f;
      sum += s[c];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv = 1.0f / sum;
#pragma unroll
    for (int c = 0; c < C; ++c) s[c] *= inv;
  } else {
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int e = c * 32 + lane;
      s[c] = (e < E) ? 1.0f / (1.0f + expf(-s[c])) : 0.0f;
    }
  }
  if (scores_out != nullptr) {
    float* srow = scores_out + (size_t)t * E;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int e = c * 32 + lane;
      if (e < E) srow[e] = s[c];
    }
  }

  int sel_e[kMaxK];
  float sel_s[kMaxK];
  if (given != nullptr) {
    // caller-fixed selection: validate range and distinctness
    for (int j = 0; j < k; ++j) {
      int e = given[(size_t)t * k + j];
      bool bad = (e < 0 || e >= E);
      for (int i = 0; i < j; ++i) bad |= (sel_e[i] == e);
      if (bad) {
        if (lane == 0) report_status(status, MOK_DEV_INVALID_ROUTING, SITE_TOPK_INDEX);
        e = 0;
      }
      sel_e[j] = e;
      // fetch score of e from its owning lane
      float v = 0.0f;
#pragma unroll
      for (int c = 0; c < C; ++c)
        if (c == (e >> 5)) v = s[c];
      sel_s[j] = __shfl_sync(0xffffffffu, v, e & 31);
    }
  } else {
    float sel[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int e = c * 32 + lane;
      sel[c] = (e < E) ? s[c] + (bias ? bias[e] : 0.0f) : -INFINITY;
    }
    unsigned taken = 0u;  // bit c: element c of this lane already selected
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY, bs = 0.0f;
      int be = 0x7fffffff;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const int e = c * 32 + lane;
        if (e < E && !((taken >> c) & 1u)) {
          if (sel[c] > bv || (sel[c] == bv && e < be)) {
            bv = sel[c];
            be = e;
            bs = s[c];
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        const float os = __shfl_xor_sync(0xffffffffu, bs, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
          bs = os;
        }
      }
      if (be < 0 || be >= E) {  // only possible with NaN scores
        if (lane == 0) report_status(status, MOK_DEV_INVALID_ROUTING, SITE_TOPK_INDEX);
        be = 0;
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      sel_e[j] = be;
      sel_s[j] = bs;
    }
  }
  float norm = 1.0f;
  if (renorm) {
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) sum += sel_s[j];
    norm = 1.0f / sum;
  }
  if (lane < k) {
    float gv = 0.0f;
    int ev = 0;
    for (int j = 0; j < k; ++j)
      if (j == lane) {
        gv = sel_s[j];
        ev = sel_e[j];
      }
    topk_idx[(size_t)t * k + lane] = ev;
    if (gates != nullptr) gates[(size_t)t * k + lane] = (renorm ? gv * norm : gv) * route_scale;
  }
}

// ----------------------------------------------------------------------------- schedule
// One CTA of 1024 threads (32 warps).  Warp w owns a contiguous chunk of assignments.
// Pass 1: per-warp histogram (warp-level match of equal experts, leader adds the count).
// Pass 2: per expert, totals, the exclusive scans (rows and 128-row tiles), and the start
//         row of each warp's share of each expert.
// Pass 3: each warp walks its chunk again in order; a lane's row is its warp's running
//         start for its expert plus the number of lower lanes with the same expert.
// The result is the stable order of assignments within each expert.
__global__ void __launch_bounds__(1024, 1)
    schedule_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ gates, int R,
                    int E, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ row_of, int32_t* __restrict__ src_of,
                    int32_t* __restrict__ tile_off, float* __restrict__ gate_row, int* status) {
  extern __shared__ int sh[];
  int* hist = sh;                 // [32][E]
  int* warp_tot = sh + 32 * E;    // [32] scan scratch
  int* warp_tot2 = warp_tot + 32; // [32]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();

  const int chunk = ((R + 31) / 32 + 31) & ~31;
  const int a_begin = min(R, warp * chunk);
  const int a_end = min(R, a_begin + chunk);
  int* my_hist = hist + warp * E;
  for (int base = a_begin; base < a_end; base += 32) {
    const int a = base + lane;
    const bool valid = a < a_end;
    int e = valid ? topk_idx[a] : -1;
    if (valid && (e < 0 || e >= E)) {
      report_status(status, MOK_DEV_INVALID_ROUTING, SITE_SCHEDULE_INDEX);
      e = 0;
    }
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(mask) - 1;
    if (valid && lane == leader) my_hist[e] += __popc(mask);
    __syncwarp();
  }
  __syncthreads();

  // totals per expert (thread e), scans over experts
  int tot = 0, tiles = 0;
  const int e = threadIdx.x;
  if (e < E) {
    for (int w = 0; w < 32; ++w) tot += hist[w * E + e];
    tiles = (tot + 127) / 128;
  }
  int inc = tot, inc2 = tiles;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    const int v2 = __shfl_up_sync(0xffffffffu, inc2, o);
    if (lane >= o) {
      inc += v;
      inc2 += v2;
    }
  }
  if (lane == 31) {
    warp_tot[warp] = inc;
    warp_tot2[warp] = inc2;
  }
  __syncthreads();
  if (warp == 0) {
    int v = warp_tot[lane], v2 = warp_tot2[lane];
    int x = v, x2 = v2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      const int y2 = __shfl_up_sync(0xffffffffu, x2, o);
      if (lane >= o) {
        x += y;
        x2 += y2;
      }
    }
    warp_tot[lane] = x - v;  // exclusive over warps
    warp_tot2[lane] = x2 - v2;
  }
  __syncthreads();
  if (e < E) {
    const int excl = warp_tot[warp] + inc - tot;
    const int excl2 = warp_tot2[warp] + inc2 - tiles;
    counts[e] = tot;
    offsets[e] = excl;
    if (tile_off) tile_off[e] = excl2;
    if (e == E - 1) {
      offsets[E] = excl + tot;
      if (tile_off) tile_off[E] = excl2 + tiles;
    }
    int run = excl;
    for (int w = 0; w < 32; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = a_begin; base < a_end; base += 32) {
    const int a = base + lane;
    const bool valid = a < a_end;
    int ex = valid ? topk_idx[a] : -1;
    if (valid && (ex < 0 || ex >= E)) ex = 0;
    const unsigned mask = __match_any_sync(0xffffffffu, ex);
    const int leader = __ffs(mask) - 1;
    if (valid) {
      const int pos = my_hist[ex] + __popc(mask & lt_mask);
      row_of[a] = pos;
      src_of[pos] = a;
      if (gate_row) gate_row[pos] = gates[a];
    }
    __syncwarp();
    if (valid && lane == leader) my_hist[ex] += __popc(mask);
    __syncwarp();
  }
}

// ----------------------------------------------------------------------------- schedule (multi-CTA)
// The same table from many CTAs, in three launches, for large T*k: the single-CTA kernel above
// walks all assignments with one CTA and grows linearly with T*k (0.35 ms at 131,072
// assignments).  Block b owns assignments [b * SCHED_CHUNK, (b + 1) * SCHED_CHUNK) and its warp
// w the 128 of them starting at w * 128:
//   1. schedule_hist_kernel: per-block histogram hist[b][e] (per-warp counts by warp match,
//      summed over the warps: integer sums, so the order of the adds does not matter);
//   2. schedule_scan_kernel (one CTA, thread e): counts, the exclusive scans over experts (rows
//      and 128-row tiles), and in place of hist[b][e] the first row of block b's share of e;
//   3. schedule_place_kernel: each block recounts its warps' shares, adds them to its block's
//      starts, and every warp walks its assignments in order as in the single-CTA kernel.
// Rows of an expert are in ascending assignment order (blocks, then warps, then lanes), the
// unique stable order, so the table is bitwise the single-CTA kernel's.
constexpr int SCHED_CHUNK = 1024;
constexpr int SCHED_THREADS = 256;
constexpr int SCHED_WARP_SPAN = SCHED_CHUNK / (SCHED_THREADS / 32);  // 128 assignments per warp

// Per-warp histogram of this block's assignments into sh[warp][E] (zeroed here).
__device__ __forceinline__ void sched_block_counts(const int32_t* __restrict__ topk_idx, int R, int E, int* sh,
                                                   int* status, bool report) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (SCHED_THREADS / 32) * E; i += SCHED_THREADS) sh[i] = 0;
  __syncthreads();
  const int a_begin = min(R, (int)blockIdx.x * SCHED_CHUNK + warp * SCHED_WARP_SPAN);
  const int a_end = min(R, a_begin + SCHED_WARP_SPAN);
  int* my = sh + warp * E;
  for (int base = a_begin; base < a_end; base += 32) {
    const int a = base + lane;
    const bool valid = a < a_end;
    int e = valid ? topk_idx[a] : -1;
    if (valid && (e < 0 || e >= E)) {
      if (report) report_status(status, MOK_DEV_INVALID_ROUTING, SITE_SCHEDULE_INDEX);
      e = 0;
    }
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    if (valid && lane == __ffs(mask) - 1) my[e] += __popc(mask);
    __syncwarp();
  }
  __syncthreads();
}

__global__ void __launch_bounds__(SCHED_THREADS)
    schedule_hist_kernel(const int32_t* __restrict__ topk_idx, int R, int E, int32_t* __restrict__ hist,
                         int* status) {
  extern __shared__ int sh[];  // [8][E]
  sched_block_counts(topk_idx, R, E, sh, status, true);
  for (int e = threadIdx.x; e < E; e += SCHED_THREADS) {
    int t = 0;
#pragma unroll
    for (int w = 0; w < SCHED_THREADS / 32; ++w) t += sh[w * E + e];
    hist[(size_t)blockIdx.x * E + e] = t;
  }
}

__global__ void __launch_bounds__(1024, 1)
    schedule_scan_kernel(int32_t* __restrict__ hist, int NB, int E, int32_t* __restrict__ counts,
                         int32_t* __restrict__ offsets, int32_t* __restrict__ tile_off) {
  __shared__ int warp_tot[32], warp_tot2[32];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int e = threadIdx.x;
  int tot = 0, tiles = 0;
  if (e < E) {
    for (int b = 0; b < NB; ++b) tot += hist[(size_t)b * E + e];
    tiles = (tot + 127) / 128;
  }
  int inc = tot, inc2 = tiles;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    const int v2 = __shfl_up_sync(0xffffffffu, inc2, o);
    if (lane >= o) {
      inc += v;
      inc2 += v2;
    }
  }
  if (lane == 31) {
    warp_tot[warp] = inc;
    warp_tot2[warp] = inc2;
  }
  __syncthreads();
  if (warp == 0) {
    const int v = warp_tot[lane], v2 = warp_tot2[lane];
    int x = v, x2 = v2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      const int y2 = __shfl_up_sync(0xffffffffu, x2, o);
      if (lane >= o) {
        x += y;
        x2 += y2;
      }
    }
    warp_tot[lane] = x - v;  // exclusive over warps
    warp_tot2[lane] = x2 - v2;
  }
  __syncthreads();
  if (e < E) {
    const int excl = warp_tot[warp] + inc - tot;
    const int excl2 = warp_tot2[warp] + inc2 - tiles;
    counts[e] = tot;
    offsets[e] = excl;
    if (tile_off) tile_off[e] = excl2;
    if (e == E - 1) {
      offsets[E] = excl + tot;
      if (tile_off) tile_off[E] = excl2 + tiles;
    }
    int run = excl;
    for (int b = 0; b < NB; ++b) {
      const int c = hist[(size_t)b * E + e];
      hist[(size_t)b * E + e] = run;
      run += c;
    }
  }
}

__global__ void __launch_bounds__(SCHED_THREADS)
    schedule_place_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ gates, int R, int E,
                          const int32_t* __restrict__ starts, int32_t* __restrict__ row_of,
                          int32_t* __restrict__ src_of, float* __restrict__ gate_row) {
  extern __shared__ int sh[];  // [8][E]
  sched_block_counts(topk_idx, R, E, sh, nullptr, false);
  for (int e = threadIdx.x; e < E; e += SCHED_THREADS) {
    int run = starts[(size_t)blockIdx.x * E + e];
#pragma unroll
    for (int w = 0; w < SCHED_THREADS / 32; ++w) {
      const int c = sh[w * E + e];
      sh[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int a_begin = min(R, (int)blockIdx.x * SCHED_CHUNK + warp * SCHED_WARP_SPAN);
  const int a_end = min(R, a_begin + SCHED_WARP_SPAN);
  int* my = sh + warp * E;
  for (int base = a_begin; base < a_end; base += 32) {
    const int a = base + lane;
    const bool valid = a < a_end;
    int ex = valid ? topk_idx[a] : -1;
    if (valid && (ex < 0 || ex >= E)) ex = 0;
    const unsigned mask = __match_any_sync(0xffffffffu, ex);
    const int leader = __ffs(mask) - 1;
    if (valid) {
      const int pos = my[ex] + __popc(mask & lt_mask);
      row_of[a] = pos;
      src_of[pos] = a;
      if (gate_row) gate_row[pos] = gates[a];
    }
    __syncwarp();
    if (valid && lane == leader) my[ex] += __popc(mask);
    __syncwarp();
  }
}

// ----------------------------------------------------------------------------- router bwd
// One warp per token.  dg_j = sum over the column-tile partials of row_of[t*k+j] (fixed
// order); then the chain rule through the gates (renormalisation) and the scores (softmax
// or sigmoid) gives the logit gradient row dl[t][0..E) (zero at unselected experts for the
// sigmoid router).
__global__ void router_dlogits_kernel(const float* __restrict__ dg_part, int n_part,
                                      const int32_t* __restrict__ row_of,
                                      const int32_t* __restrict__ topk_idx,
                                      const float* __restrict__ gates,
                                      const float* __restrict__ scores, int T, int E, int k,
                                      int router, int renorm, float route_scale,
                                      float* __restrict__ dgates_out, float* __restrict__ dl) {
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float my_dg = 0.0f;
  int my_e = -1;
  float my_s = 0.0f, my_g = 0.0f;
  if (lane < k) {
    const int row = row_of[(size_t)t * k + lane];
    const float* p = dg_part + (size_t)row * n_part;
    for (int q = 0; q < n_part; ++q) my_dg += p[q];
    my_e = topk_idx[(size_t)t * k + lane];
    my_s = scores[(size_t)t * E + my_e];
    my_g = gates[(size_t)t * k + lane];
    if (dgates_out) dgates_out[(size_t)t * k + lane] = my_dg;
  }
  // broadcast selected values; sums in j order on every lane
  float dsum = 0.0f, ssum = 0.0f;
  float dg_j[kMaxK], s_j[kMaxK];
  int e_j[kMaxK];
  for (int j = 0; j < k; ++j) {
    dg_j[j] = __shfl_sync(0xffffffffu, my_dg, j);
    s_j[j] = __shfl_sync(0xffffffffu, my_s, j);
    e_j[j] = __shfl_sync(0xffffffffu, my_e, j);
    const float gj = __shfl_sync(0xffffffffu, my_g, j);
    dsum = fmaf(dg_j[j], gj, dsum);
    ssum += s_j[j];
  }
  // d loss / d score at selected expert j
  float ds_j[kMaxK];
  for (int j = 0; j < k; ++j)
    ds_j[j] = renorm ? (route_scale * dg_j[j] - dsum) / ssum : route_scale * dg_j[j];
  float* dlrow = dl + (size_t)t * E;
  if (router == 1) {
    for (int e0 = lane; e0 < E; e0 += 32) dlrow[e0] = 0.0f;
    __syncwarp();
    if (lane < k) {
      float dsv = 0.0f;
      for (int j = 0; j < k; ++j)
        if (j == lane) dsv = ds_j[j];
      dlrow[my_e] = dsv * my_s * (1.0f - my_s);
    }
  } else {
    // softmax: dl_i = p_i * (ds_i [i selected] - sum_m ds_m p_m)
    float dot = 0.0f;
    for (int j = 0; j < k; ++j) dot = fmaf(ds_j[j], s_j[j], dot);
    for (int e0 = lane; e0 < E; e0 += 32) {
      float dsi = 0.0f;
      for (int j = 0; j < k; ++j)
        if (e_j[j] == e0) dsi = ds_j[j];
      const float p = scores[(size_t)t * E + e0];
      dlrow[e0] = p * (dsi - dot);
    }
  }
}

// dW_r[e][h] = sum over tokens t (ascending) of dl[t][e] * x[t][h], fp32.
// Sigmoid router: dl[t][e] is nonzero only where t selected e, i.e. on the rows of expert
// e's segment (ascending tokens).  Softmax: all tokens.  Block = (expert, 2048 columns).
__global__ void __launch_bounds__(256)
    router_wgrad_kernel(const float* __restrict__ dl, const __nv_bfloat16* __restrict__ x,
                        const int32_t* __restrict__ offsets, const int32_t* __restrict__ src_of,
                        int T, int H, int E, int k, int sparse, float* __restrict__ dw) {
  __shared__ int s_tok[256];
  __shared__ float s_coef[256];
  const int e = blockIdx.x;
  const int h0 = blockIdx.y * 2048 + threadIdx.x * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  const int n = sparse ? (offsets[e + 1] - offsets[e]) : T;
  const int r0 = sparse ? offsets[e] : 0;
  for (int base = 0; base < n; base += 256) {
    const int i = base + threadIdx.x;
    if (i < n) {
      const int tok = sparse ? src_of[r0 + i] / k : i;
      s_tok[threadIdx.x] = tok;
      s_coef[threadIdx.x] = dl[(size_t)tok * E + e];
    }
    __syncthreads();
    const int m = min(256, n - base);
    if (h0 < H) {
      for (int q = 0; q < m; ++q) {
        const float c = s_coef[q];
        const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)s_tok[q] * H + h0);
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(b[j]);
          acc[2 * j] = fmaf(c, f.x, acc[2 * j]);
          acc[2 * j + 1] = fmaf(c, f.y, acc[2 * j + 1]);
        }
      }
    }
    __syncthreads();
  }
  if (h0 < H) {
    float4* out = reinterpret_cast<float4*>(dw + (size_t)e * H + h0);
    out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// ----------------------------------------------------------------------------- ring tables
// Minibatch mb holds the sorted rows [mb*m, mb*m + rows_mb).  One CTA per minibatch (threads
// over experts) cuts the expert segments at its edges: mb_off[mb][e] = clamp(offsets[e] - r0,
// 0, rows_mb), and scans the chunks of at most tile_rows rows of each cut segment into mb_toff[mb][e];
// mb_tiles[mb] = total chunks * n_tiles (the column tiles of GEMM1).
__global__ void __launch_bounds__(1024)
    mb_tables_kernel(const int32_t* __restrict__ offsets, int E, int R, int m, int n_tiles, int tile_rows,
                     int32_t* __restrict__ mb_off, int32_t* __restrict__ mb_toff, int32_t* __restrict__ mb_tiles) {
  __shared__ int warp_tot[32];
  const int mb = blockIdx.x;
  const int r0 = mb * m;
  const int rows = min(m, R - r0);
  const int e = threadIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tiles = 0;
  if (e < E) {
    const int lo = min(max(offsets[e] - r0, 0), rows);
    const int hi = min(max(offsets[e + 1] - r0, 0), rows);
    tiles = (hi - lo + tile_rows - 1) / tile_rows;
    mb_off[(size_t)mb * (E + 1) + e] = lo;
  }
  if (e == 0) mb_off[(size_t)mb * (E + 1) + E] = min(max(offsets[E] - r0, 0), rows);
  int inc = tiles;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int v = warp_tot[lane];
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    warp_tot[lane] = x - v;
  }
  __syncthreads();
  const int excl = warp_tot[warp] + inc - tiles;
  if (e < E) mb_toff[(size_t)mb * (E + 1) + e] = excl;
  if (e == E - 1) {
    mb_toff[(size_t)mb * (E + 1) + E] = excl + tiles;
    mb_tiles[mb] = (excl + tiles) * n_tiles;
  }
}

// mb_start = exclusive prefix of mb_tiles (n_mb + 1 entries), one thread, fixed order.
__global__ void mb_start_kernel(const int32_t* __restrict__ mb_tiles, int n_mb, int32_t* __restrict__ mb_start) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < n_mb; ++i) {
      mb_start[i] = run;
      run += mb_tiles[i];
    }
    mb_start[n_mb] = run;
  }
}

// ----------------------------------------------------------------------------- launchers
cudaError_t launch_mb_tables(const int32_t* offsets, int E, int R, int m, int n_mb, int n_tiles, int tile_rows, int32_t* mb_off,
                             int32_t* mb_toff, int32_t* mb_tiles, int32_t* mb_start, cudaStream_t st) {
  mb_tables_kernel<<<n_mb, 1024, 0, st>>>(offsets, E, R, m, n_tiles, tile_rows, mb_off, mb_toff, mb_tiles);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  mb_start_kernel<<<1, 32, 0, st>>>(mb_tiles, n_mb, mb_start);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, const float* bias, const int32_t* given, int T, int E,
                        int k, int router, int renorm, float route_scale, int32_t* topk_idx,
                        float* gates, float* scores, int* status, cudaStream_t st) {
  const int warps = 8;
  const dim3 grid((T + warps - 1) / warps), block(warps * 32);
#define MOK_TOPK(CC)                                                                                          \
  topk_kernel<CC><<<grid, block, 0, st>>>(logits, bias, given, T, E, k, router, renorm, route_scale, topk_idx, \
                                          gates, scores, status)
  if (E <= 32) MOK_TOPK(1);
  else if (E <= 64) MOK_TOPK(2);
  else if (E <= 128) MOK_TOPK(4);
  else if (E <= 256) MOK_TOPK(8);
  else if (E <= 512) MOK_TOPK(16);
  else MOK_TOPK(32);
#undef MOK_TOPK
  return cudaGetLastError();
}

cudaError_t launch_schedule(const int32_t* topk_idx, const float* gates, int R, int E, int32_t* counts,
                            int32_t* offsets, int32_t* row_of, int32_t* src_of, int32_t* tile_off,
                            float* gate_row, int* status, cudaStream_t st) {
  const size_t smem = (size_t)(32 * E + 64) * sizeof(int);
  cudaError_t err = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         32 * kMaxE * 4 + 64 * 4);
  if (err != cudaSuccess) return err;
  schedule_kernel<<<1, 1024, smem, st>>>(topk_idx, gates, R, E, counts, offsets, row_of, src_of, tile_off,
                                         gate_row, status);
  return cudaGetLastError();
}

cudaError_t launch_router_dlogits(const float* dg_part, int n_part, const int32_t* row_of,
                                  const int32_t* topk_idx, const float* gates, const float* scores, int T,
                                  int E, int k, int router, int renorm, float route_scale, float* dgates,
                                  float* dl, cudaStream_t st) {
  const int warps = 8;
  router_dlogits_kernel<<<(T + warps - 1) / warps, warps * 32, 0, st>>>(
      dg_part, n_part, row_of, topk_idx, gates, scores, T, E, k, router, renorm, route_scale, dgates, dl);
  return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const float* dl, const void* x, const int32_t* offsets, const int32_t* src_of,
                                int T, int H, int E, int k, int sparse, float* dw, cudaStream_t st) {
  dim3 grid(E, (H + 2047) / 2048);
  router_wgrad_kernel<<<grid, 256, 0, st>>>(dl, reinterpret_cast<const __nv_bfloat16*>(x), offsets, src_of, T,
                                            H, E, k, sparse, dw);
  return cudaGetLastError();
}

int schedule_blocks(int R) { return (R + SCHED_CHUNK - 1) / SCHED_CHUNK; }

cudaError_t launch_schedule_multi(const int32_t* topk_idx, const float* gates, int R, int E, int32_t* counts,
                                  int32_t* offsets, int32_t* row_of, int32_t* src_of, int32_t* tile_off,
                                  float* gate_row, int32_t* hist, int* status, cudaStream_t st) {
  const int NB = schedule_blocks(R);
  const size_t smem = (size_t)(SCHED_THREADS / 32) * E * sizeof(int);
  if (NB > 0) {
    schedule_hist_kernel<<<NB, SCHED_THREADS, smem, st>>>(topk_idx, R, E, hist, status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  schedule_scan_kernel<<<1, 1024, 0, st>>>(hist, NB, E, counts, offsets, tile_off);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || NB == 0) return err;
  schedule_place_kernel<<<NB, SCHED_THREADS, smem, st>>>(topk_idx, gates, R, E, hist, row_of, src_of, gate_row);
  return cudaGetLastError();
}

}  // namespace mok
