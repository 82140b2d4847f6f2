// Persistent tcgen05 GEMM for the expert-grouped products of one MoE layer (sm_103a).
//
// One CTA per SM, 6 warps:
//   warp 0      TMA producer: loads A and B tiles of 64 K-elements into a ring of stages
//   warp 1      MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16 -> f32) into TMEM, 128 x BN tile
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, fused elementwise work, stores
// The accumulator is double-buffered in TMEM (2 x BN columns), so the epilogue of tile i
// overlaps the main loop of tile i+1.  Tiles are dealt round-robin over the CTAs in a fixed
// order; every output element is owned by one tile and reduced over K in a fixed order, so
// results do not depend on timing.
//
// Split operands: an operand produced by this layer (SwiGLU output, its gradient) is kept as
// a pair of bf16 tensors hi + lo with lo = bf16(v - hi), about 16 significant bits.  The MMA
// warp issues hi and lo products into the same fp32 accumulator, so the GEMM sees the operand
// at nearly fp32 precision while the tensor cores stay on the bf16 path.
//
// Modes (how A, B and the tiles are laid out):
//   MODE_DENSE  A [M][K], B [N][K], both K-major                  (router logits)
//   MODE_ROWS   A = expert-sorted rows [R][K] (K-major), B [E][N][K] K-major
//               (GEMM1 x_g W13^T with SwiGLU, GEMM2 a W2^T)
//   MODE_DGRAD  A = rows [R][K] K-major, B [E][K][N] (N contiguous: MN-major)
//               (dA' = dY_g W2[e], dX_g = dHU W13[e])
//   MODE_WGRAD  A = rows [R][M] and B = rows [R][N], both MN-major; K runs over the rows of
//               one expert; output stored transposed, out[e][n][m], so that the 32 lanes of a
//               warp (32 consecutive m) write 32 consecutive elements
// Rows of one expert are contiguous (the schedule table); a 128-row tile that runs past its
// expert reads the next expert's rows (discarded at the store) or TMA zero fill past R.
// In MODE_WGRAD the rows past the expert's end inside the last K block are zeroed in shared
// memory before the MMA reads them.
#pragma once
#include <cuda_bf16.h>

#include "mx.cuh"
#include "ptx.cuh"

namespace mok {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int GEMM_THREADS = 192;
constexpr int A_TILE = BM * BK * 2;      // 16 KB
constexpr int SMEM_RING = 192 * 1024;    // bytes for the stage ring
constexpr int MN_ATOM_BYTES = 64 * 128;  // one MN-major 128B-swizzle atom column: 64 K rows x 128 B

// Leading / stride byte offsets of the MN-major 128B-swizzled operand layout:
// LBO = distance between 64-element MN atom columns, SBO = distance between 8-row K groups.
#ifndef MOK_MN_LBO
#define MOK_MN_LBO MN_ATOM_BYTES
#endif
#ifndef MOK_MN_SBO
#define MOK_MN_SBO 1024
#endif

// MODE_RING: GEMM1 of the ring forward.  A = the token ring (bf16 [slots * mb_rows][H]);
// CTAs [0, comm_ctas) gather expert-sorted rows into ring slots minibatch by minibatch, the
// other CTAs run the minibatches' grouped-GEMM tiles in minibatch order.  A minibatch's
// tiles wait until its rows are gathered (counter `gathered`); a slot is refilled only after
// every tile of the minibatch it held has finished (counter `consumed`).
enum GemmMode { MODE_DENSE = 0, MODE_ROWS = 1, MODE_DGRAD = 2, MODE_WGRAD = 3, MODE_RING = 4 };
// EPI_SWIGLU_PAIRED (narrow kernel only): SwiGLU with the gate and up rows of the same
// intermediate indices in two MMAs sharing the row operand, h and u in one thread's TMEM columns.
// EPI_F32_PAIRED (narrow kernel only): two weight tiles 256 rows apart in two MMAs sharing the row
// operand, accumulated in columns [0, N) and [256, 256 + N).
enum GemmEpi {
  EPI_F32 = 0,
  EPI_SWIGLU = 2,
  EPI_SWIGLU_BWD = 3,
  EPI_T_F32 = 4,
  EPI_T_BF16 = 5,
  EPI_SWIGLU_PAIRED = 7,
  EPI_F32_PAIRED = 8  // narrow kernel only: two 256-row weight tiles per pair tile, fp32 out
};
enum GemmSplit { SPLIT_NONE = 0, SPLIT_A = 1, SPLIT_B = 2 };

struct GemmArgs {
  int M;            // DENSE: rows of A; WGRAD: output rows per expert (the contiguous output dim)
  int N;            // output columns (per expert); SWIGLU: I (the tile pairs gate and up)
  int K;            // reduction length (DENSE / ROWS / DGRAD)
  int E;            // experts (groups)
  int I;            // SWIGLU / SWIGLU_BWD: intermediate width
  int total_tiles;  // host-known tile count, or -1: tile_off[E] * n_tiles (grouped rows)
  const int* offsets;   // [E+1] expert row offsets
  const int* tile_off;  // [E+1] prefix of ceil(rows/128)
  void* out0;
  void* out1;
  void* out2;
  void* out3;
  void* out4;
  long long ld0, ld1, ld2;
  int f16;                  // narrow kernels: the MMA operands are fp16 (else bf16)
  int a_f16;                // narrow SwiGLU epilogues: a = silu(h) u stored as one fp16 value in out1
                            // (11 significant bits) instead of a bf16 hi / lo pair
  const float* hu;          // SWIGLU_BWD: saved h | u (fp32)
  const float* gate_row;    // SWIGLU_BWD: gate of each row
  int* status;
  // MODE_RING
  int comm_ctas;            // gathering CTAs (the first ones of the grid)
  int n_mb;                 // minibatches
  int mb_rows;              // rows per minibatch (the last one may be shorter)
  int ring_slots;           // minibatches the ring holds
  int ring_shift;           // minibatch mb lives in slot (mb + ring_shift) % ring_slots
  int R;                    // all rows
  int k_top;                // experts per token (row r holds token src_of[r] / k_top)
  int H;
  const int* mb_off;        // [n_mb][E+1] expert row offsets inside each minibatch
  const int* mb_toff;       // [n_mb][E+1] prefix of m-tiles inside each minibatch
  const int* mb_start;      // [n_mb+1] first tile of each minibatch
  int* gathered;            // [n_mb] rows gathered
  int* consumed;            // [n_mb] epilogue warps finished (consume_per_tile per tile)
  int consume_per_tile;     // epilogue warps counting out one tile (4, or 8 for a CTA pair)
  int* ticket;              // narrow ring GEMM1 / GEMM2: next tile to take (one counter for all pairs)
  int fence_out;            // ring GEMM1: make each tile's outputs visible before counting it consumed
  int mb_tiles1;            // ring GEMM2: GEMM1 tiles per row chunk (the minibatch tables count those)
  int* done;                // ring GEMM2: epilogue warps finished, for the combine
  const __nv_bfloat16* x;   // [T][H] tokens
  const int* src_of;        // [R]
  __nv_bfloat16* ring;      // [ring_slots * mb_rows][H]
};

// GemmArgs with the fields every launch sets (the rest zero).
inline GemmArgs base_args(int E, const int32_t* offsets, const int32_t* tile_off, int* status) {
  GemmArgs g{};
  g.E = E;
  g.offsets = offsets;
  g.tile_off = tile_off;
  g.total_tiles = -1;
  g.status = status;
  return g;
}

struct TileInfo {
  int e, m, n;
  int row0;   // first A row (ROWS/DGRAD/DENSE) or first K row (WGRAD)
  int rows;   // valid output rows (ROWS/DGRAD/DENSE) or K rows (WGRAD)
  int nkb;    // K blocks
  int mt;     // ROWS/DGRAD: number of 128-row tiles of this expert (they share each weight tile)
  int mb;     // RING: minibatch of the tile (row0 / rows are inside the minibatch)
};

template <int MODE, int EPI, int SPLIT, int BN_>
struct GemmCfg {
  static constexpr int BN = BN_;
  static constexpr bool kAmn = (MODE == MODE_WGRAD);
  static constexpr bool kBmn = (MODE == MODE_DGRAD || MODE == MODE_WGRAD);
  static constexpr int B_TILE = BN * BK * 2;
  static constexpr int A_TILES = SPLIT == SPLIT_A ? 2 : 1;
  static constexpr int B_TILES = SPLIT == SPLIT_B ? 2 : 1;
  static constexpr int STAGE_BYTES = A_TILE * A_TILES + B_TILE * B_TILES;
  static constexpr int TX_BYTES = STAGE_BYTES;  // bytes TMA delivers into one stage
  static constexpr int THREADS = 192;
  // WGRAD stages its 32 x 32 output blocks in shared memory for TMA stores: one buffer of up
  // to 32 x 32 fp32 per block of a tile, per epilogue warp.
  // ROWS / DGRAD fp32 and SwiGLU outputs leave through TMA stores from one 4 KB buffer per
  // epilogue warp
  static constexpr bool kTmaEpi = (MODE == MODE_ROWS || MODE == MODE_DGRAD) && (EPI == EPI_F32 || EPI == EPI_SWIGLU);
  static constexpr int STG_BYTES = (MODE == MODE_WGRAD)                        ? 4 * (BN / 32) * 4096
                                   : (kTmaEpi || EPI == EPI_SWIGLU_BWD) ? 4 * 4096
                                                                        : 0;
  static constexpr int RING = (MODE == MODE_WGRAD) ? 3 * STAGE_BYTES : SMEM_RING;
  // the router GEMM (MODE_DENSE, 64-column tiles of 24 KB stages) walks its whole K = H per tile:
  // more stages in flight keep its loads' latency covered (at most 8: the barriers' 256 bytes)
  static constexpr int MAX_STAGES = MODE == MODE_DENSE ? 8 : 4;
  static constexpr int STAGES = (RING / STAGE_BYTES) < MAX_STAGES ? (RING / STAGE_BYTES) : MAX_STAGES;
  static_assert((2 * STAGES + 5) * 8 + 8 <= 256, "barriers, TMEM address and abort flag");
  static constexpr int RINGS_BYTES = STAGES * STAGE_BYTES;
  static constexpr int ACC_COLS = BN;
  static constexpr int TMEM_COLS = 2 * BN;
  static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                "tcgen05.alloc takes a power of two from 32 to 512 columns");
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, kAmn, kBmn);
  static __host__ __device__ int n_tiles(const GemmArgs& a) {
    return EPI == EPI_SWIGLU ? a.I / 128 : (a.N + BN - 1) / BN;
  }
  static __host__ __device__ constexpr size_t smem_bytes(int E) {
    return size_t(RINGS_BYTES) + STG_BYTES + 1024 /*align*/ + 256 /*barriers*/ + size_t(2) * (E + 1) * 4;
  }
};

template <int MODE, int EPI, int SPLIT, int BN_>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, int g, const int* s_off, const int* s_toff) {
  using C = GemmCfg<MODE, EPI, SPLIT, BN_>;
  TileInfo t;
  const int NT = C::n_tiles(a);
  if (MODE == MODE_DENSE) {
    const int MT = (a.M + BM - 1) / BM;
    t.e = 0;
    t.m = g % MT;
    t.n = g / MT;
    t.row0 = t.m * BM;
    t.rows = min(BM, a.M - t.row0);
    t.nkb = a.K / BK;
    t.mt = MT;
  } else if (MODE == MODE_WGRAD) {
    const int MT = a.M / BM;
    const int per_e = MT * NT;
    t.e = g / per_e;
    const int rem = g - t.e * per_e;
    t.n = rem / MT;  // m fastest: neighbouring CTAs share the B (N) columns of the expert
    t.m = rem - t.n * MT;
    t.row0 = s_off[t.e];
    t.rows = s_off[t.e + 1] - t.row0;
    t.nkb = (t.rows + BK - 1) / BK;
    t.mt = MT;
  } else if (MODE == MODE_RING) {
    // minibatch: largest mb with mb_start[mb] <= g; then the grouped decode inside it
    int lo = 0, hi = a.n_mb;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(&a.mb_start[mid]) <= g) lo = mid; else hi = mid;
    }
    t.mb = lo;
    const int* toff = a.mb_toff + (size_t)lo * (a.E + 1);
    const int* off = a.mb_off + (size_t)lo * (a.E + 1);
    const int gl = g - __ldg(&a.mb_start[lo]);
    int el = 0, eh = a.E;
    while (eh - el > 1) {
      const int mid = (el + eh) >> 1;
      if (__ldg(&toff[mid]) * NT <= gl) el = mid; else eh = mid;
    }
    t.e = el;
    const int Me = __ldg(&toff[el + 1]) - __ldg(&toff[el]);
    const int local = gl - __ldg(&toff[el]) * NT;
    t.n = local / Me;
    t.m = local - t.n * Me;
    t.row0 = __ldg(&off[el]) + t.m * BM;
    t.rows = min(BM, __ldg(&off[el + 1]) - t.row0);
    t.nkb = a.K / BK;
    t.mt = Me;
  } else {
    // expert e owns tiles [tile_off[e]*NT, tile_off[e+1]*NT); inside, m runs fastest so the
    // m-tiles of one expert that share a weight tile are dealt to neighbouring CTAs.
    int lo = 0, hi = a.E;  // largest e with s_toff[e]*NT <= g (the last of equal starts owns tiles)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_toff[mid] * NT <= g) lo = mid; else hi = mid;
    }
    t.e = lo;
    const int Me = s_toff[lo + 1] - s_toff[lo];
    const int local = g - s_toff[lo] * NT;
    t.n = local / Me;
    t.m = local - t.n * Me;
    t.row0 = s_off[lo] + t.m * BM;
    t.rows = min(BM, s_off[lo + 1] - t.row0);
    t.nkb = a.K / BK;
    t.mt = Me;
  }
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// hi = bf16(v), lo = bf16(v - hi) for a pair of values.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

__device__ __forceinline__ void store_u32x16(void* dst, const uint32_t (&p)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j) d[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Waits (one thread) until *p >= target; bounded like the mbarrier waits.
__device__ __forceinline__ bool wait_counter(const int* p, int target, int* status, int site) {
  if (ld_acquire_gpu(p) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (ld_acquire_gpu(p) >= target) return true;
    __nanosleep(64);
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      report_status(status, MOK_DEV_TIMEOUT, site);
      return false;
    }
  }
}

// Epilogue of one accumulator row (this thread's TMEM lane) of a 128 x BN tile: fp32 output
// row, columns n*BN .. n*BN+BN-1 (clipped at args.N).
template <int BN>
__device__ __forceinline__ void epi_f32_row(uint32_t tacc, bool valid, long long row, int n, const GemmArgs& args) {
  float* out = reinterpret_cast<float*>(args.out0) + row * args.ld0;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tacc + c * 32, v);
    tmem_wait_ld();
    const int col0 = n * BN + c * 32;
    if (valid) {
      if (col0 + 32 <= args.N) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(out + col0 + j) = make_float4(
              __uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < args.N) out[col0 + j] = __uint_as_float(v[j]);
      }
    }
  }
}

// SwiGLU epilogue of one accumulator row: columns 0..127 are the gate projection h, 128..255
// the up projection u, for intermediate indices n*128 .. n*128+127.  Stores h | u in fp32 and
// a = silu(h) u as a bf16 hi / lo pair.
__device__ __forceinline__ void epi_swiglu_row(uint32_t tacc, bool valid, long long row, int n,
                                               const GemmArgs& args) {
  float* hu = reinterpret_cast<float*>(args.out0) + row * args.ld0;
  __nv_bfloat16* act_hi = reinterpret_cast<__nv_bfloat16*>(args.out1) + row * args.ld1;
  __nv_bfloat16* act_lo = reinterpret_cast<__nv_bfloat16*>(args.out2) + row * args.ld1;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t vh[32], vu[32];
    tmem_ld_32x32b_x32(tacc + c * 32, vh);
    tmem_ld_32x32b_x32(tacc + 128 + c * 32, vu);
    tmem_wait_ld();
    if (valid) {
      const int col = n * 128 + c * 32;
      uint32_t phi[16], plo[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float h0 = __uint_as_float(vh[2 * j]), h1 = __uint_as_float(vh[2 * j + 1]);
        const float u0 = __uint_as_float(vu[2 * j]), u1 = __uint_as_float(vu[2 * j + 1]);
        const float a0 = h0 / (1.0f + __expf(-h0)) * u0;
        const float a1 = h1 / (1.0f + __expf(-h1)) * u1;
        split_bf16x2(a0, a1, phi[j], plo[j]);
      }
      float4* dh = reinterpret_cast<float4*>(hu + col);
      float4* du = reinterpret_cast<float4*>(hu + args.I + col);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        dh[j] = make_float4(__uint_as_float(vh[4 * j]), __uint_as_float(vh[4 * j + 1]), __uint_as_float(vh[4 * j + 2]),
                            __uint_as_float(vh[4 * j + 3]));
        du[j] = make_float4(__uint_as_float(vu[4 * j]), __uint_as_float(vu[4 * j + 1]), __uint_as_float(vu[4 * j + 2]),
                            __uint_as_float(vu[4 * j + 3]));
      }
      store_u32x16(act_hi + col, phi);
      store_u32x16(act_lo + col, plo);
    }
  }
}

// ---------------------------------------------------------------- epilogues through TMA stores
// A warp owns 32 accumulator rows (its TMEM lane quarter).  When all 32 rows are valid, a
// 32 x 32 block leaves through shared memory and one TMA tile store (full lines, no per-thread
// scattered stores competing with the operand traffic of the main loop); a warp whose rows
// cross the end of the expert's segment stores its valid rows directly, so that no row of
// another expert is touched.

// fp32 block (thread = row r, v = its 32 columns) into a 128B-swizzled 32 x 128 B buffer
// (1024-byte aligned): 16-byte chunk c of row r sits at r*128 + ((c ^ (r % 8)) * 16).
__device__ __forceinline__ void stage_f32_sw128(uint8_t* stg, const uint32_t (&v)[32], int lane) {
  uint8_t* row = stg + lane * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// bf16 block (thread = row r, p = its 16 packed pairs) into a 64B-swizzled 32 x 64 B buffer
// (512-byte aligned): 16-byte chunk c of row r sits at r*64 + ((c ^ ((r / 2) % 4)) * 16).
__device__ __forceinline__ void stage_bf16_sw64(uint8_t* stg, const uint32_t (&p)[16], int lane) {
  uint8_t* row = stg + lane * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(row + ((c ^ ((lane >> 1) & 3)) << 4)) = make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
}

// fp32 output rows through TMA stores.  `stg`: this warp's 4 KB buffer; `row0`: first row of
// the warp's 32; `nvalid`: how many of them are valid; tmO: [rows][N] fp32, box 32 x 32, SW128.
template <int BN>
__device__ __forceinline__ void epi_f32_tma(uint32_t tacc, long long row0, int nvalid, int n, const GemmArgs& args,
                                            const CUtensorMap* tmO, uint8_t* stg, int lane) {
  if (nvalid < 32) {
    epi_f32_row<BN>(tacc, lane < nvalid, row0 + lane, n, args);
    return;
  }
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tacc + c * 32, v);
    tmem_wait_ld();
    const int col0 = n * BN + c * 32;
    if (col0 >= args.N) continue;
    if (lane == 0) bulk_wait_group_read<0>();  // the previous block has left the buffer
    __syncwarp();
    stage_f32_sw128(stg, v, lane);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmO, smem_u32(stg), col0, (int)row0);
      bulk_commit_group();
    }
  }
}

// SwiGLU epilogue through TMA stores: h | u fp32 (tmHU: [rows][2I], box 32 x 32, SW128) and
// a as hi / lo bf16 (tmAh, tmAl: [rows][I], box 32 x 32, SW64).  `stg`: this warp's buffer,
// 1024-byte aligned: 12 KB (h 4 KB, u 4 KB, a hi 2 KB, a lo 2 KB, all four in flight) when
// SEPARATE, else 4 KB that the four blocks pass through one after another.
template <bool SEPARATE>
__device__ __forceinline__ void epi_swiglu_tma(uint32_t tacc, long long row0, int nvalid, int n, const GemmArgs& args,
                                               const CUtensorMap* tmHU, const CUtensorMap* tmAh,
                                               const CUtensorMap* tmAl, uint8_t* stg, int lane) {
  if (nvalid < 32) {
    epi_swiglu_row(tacc, lane < nvalid, row0 + lane, n, args);
    return;
  }
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t vh[32], vu[32];
    tmem_ld_32x32b_x32(tacc + c * 32, vh);
    tmem_ld_32x32b_x32(tacc + 128 + c * 32, vu);
    tmem_wait_ld();
    uint32_t phi[16], plo[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float h0 = __uint_as_float(vh[2 * j]), h1 = __uint_as_float(vh[2 * j + 1]);
      const float u0 = __uint_as_float(vu[2 * j]), u1 = __uint_as_float(vu[2 * j + 1]);
      const float a0 = h0 / (1.0f + __expf(-h0)) * u0;
      const float a1 = h1 / (1.0f + __expf(-h1)) * u1;
      split_bf16x2(a0, a1, phi[j], plo[j]);
    }
    const int col = n * 128 + c * 32;
    if (SEPARATE) {
      if (lane == 0) bulk_wait_group_read<0>();
      __syncwarp();
      stage_f32_sw128(stg, vh, lane);
      stage_f32_sw128(stg + 4096, vu, lane);
      stage_bf16_sw64(stg + 8192, phi, lane);
      stage_bf16_sw64(stg + 10240, plo, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmHU, smem_u32(stg), col, (int)row0);
        tma_store_2d(tmHU, smem_u32(stg + 4096), args.I + col, (int)row0);
        tma_store_2d(tmAh, smem_u32(stg + 8192), col, (int)row0);
        tma_store_2d(tmAl, smem_u32(stg + 10240), col, (int)row0);
        bulk_commit_group();
      }
    } else {
#pragma unroll
      for (int piece = 0; piece < 4; ++piece) {
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        if (piece == 0) stage_f32_sw128(stg, vh, lane);
        else if (piece == 1) stage_f32_sw128(stg, vu, lane);
        else stage_bf16_sw64(stg, piece == 2 ? phi : plo, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (piece == 0) tma_store_2d(tmHU, smem_u32(stg), col, (int)row0);
          else if (piece == 1) tma_store_2d(tmHU, smem_u32(stg), args.I + col, (int)row0);
          else tma_store_2d(piece == 2 ? tmAh : tmAl, smem_u32(stg), col, (int)row0);
          bulk_commit_group();
        }
      }
    }
  }
}

// SwiGLU backward epilogue with the columns on the lanes.  The accumulator dA' = dY_g W2[e] comes
// out of TMEM one row per thread; each 32 x 32 block goes through a 128B-swizzled 4 KB buffer and
// is read back so that 8 lanes share a row and each lane takes 4 consecutive columns: the loads
// of h | u (16 bytes a lane) and the six bf16 outputs (dh, du, g*a as hi / lo; 8 bytes a lane)
// then touch 4 rows per instruction instead of 32.  out0/out1: dh|du hi/lo [R][2I]; out2/out3:
// g*a hi/lo [R][I]; out4: the row's partial gate gradient <dA', a> over this tile's columns.
__device__ __forceinline__ uint2 pack_bf16x4(const float (&v)[4]) {
  return make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
}

template <int BN>
__device__ __forceinline__ void epi_swiglu_bwd_cols(uint32_t tacc, long long row0, int nvalid, int n,
                                                    const GemmArgs& args, uint8_t* stg, int lane) {
  const int I = args.I;
  const int sub = lane >> 3;   // row within each group of 4
  const int q = lane & 7;      // 4-column group within the 32-column block
  const float g_lane = lane < nvalid ? args.gate_row[row0 + lane] : 0.0f;  // gate of row `lane`
  float dgacc[8];              // rows sub, sub+4, ..., sub+28
#pragma unroll
  for (int i = 0; i < 8; ++i) dgacc[i] = 0.0f;
  __nv_bfloat16* dhu_hi = reinterpret_cast<__nv_bfloat16*>(args.out0);
  __nv_bfloat16* dhu_lo = reinterpret_cast<__nv_bfloat16*>(args.out1);
  __nv_bfloat16* ga_hi = reinterpret_cast<__nv_bfloat16*>(args.out2);
  __nv_bfloat16* ga_lo = reinterpret_cast<__nv_bfloat16*>(args.out3);
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    if (n * BN + c * 32 >= I) break;  // the tile reaches past I (I a multiple of 128, not 256)
    const int col = n * BN + c * 32 + 4 * q;
    // this block's h | u first: their latency overlaps the TMEM load and the transpose
    float4 h4s[8], u4s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + sub;
      if (r < nvalid) {
        const long long row = row0 + r;
        h4s[i] = *reinterpret_cast<const float4*>(args.hu + row * 2 * I + col);
        u4s[i] = *reinterpret_cast<const float4*>(args.hu + row * 2 * I + I + col);
      } else {
        h4s[i] = u4s[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
    uint32_t v[32];
    tmem_ld_32x32b_x32(tacc + c * 32, v);
    tmem_wait_ld();
    __syncwarp();  // the previous block has been read back
    stage_f32_sw128(stg, v, lane);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + sub;
      const float g = __shfl_sync(0xffffffffu, g_lane, r);
      if (r < nvalid) {
        const float4 dap4 = *reinterpret_cast<const float4*>(stg + r * 128 + ((q ^ (r & 7)) << 4));
        const long long row = row0 + r;
        const float4 h4 = h4s[i];
        const float4 u4 = u4s[i];
        const float dap[4] = {dap4.x, dap4.y, dap4.z, dap4.w};
        const float hv[4] = {h4.x, h4.y, h4.z, h4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
        float dh[4], du[4], ga[4], dh_l[4], du_l[4], ga_l[4];
#pragma unroll
        for (int z = 0; z < 4; ++z) {
          const float sg = __fdividef(1.0f, 1.0f + __expf(-hv[z]));
          const float sl = hv[z] * sg;
          const float a = sl * uv[z];
          dgacc[i] = fmaf(dap[z], a, dgacc[i]);
          const float dA = g * dap[z];
          const float vdh = dA * uv[z] * sg * (1.0f + hv[z] * (1.0f - sg));
          const float vdu = dA * sl;
          const float vga = g * a;
          dh[z] = __bfloat162float(__float2bfloat16_rn(vdh));
          du[z] = __bfloat162float(__float2bfloat16_rn(vdu));
          ga[z] = __bfloat162float(__float2bfloat16_rn(vga));
          dh_l[z] = vdh - dh[z];
          du_l[z] = vdu - du[z];
          ga_l[z] = vga - ga[z];
        }
        *reinterpret_cast<uint2*>(dhu_hi + row * args.ld0 + col) = pack_bf16x4(dh);
        *reinterpret_cast<uint2*>(dhu_lo + row * args.ld0 + col) = pack_bf16x4(dh_l);
        *reinterpret_cast<uint2*>(dhu_hi + row * args.ld0 + I + col) = pack_bf16x4(du);
        *reinterpret_cast<uint2*>(dhu_lo + row * args.ld0 + I + col) = pack_bf16x4(du_l);
        *reinterpret_cast<uint2*>(ga_hi + row * args.ld1 + col) = pack_bf16x4(ga);
        *reinterpret_cast<uint2*>(ga_lo + row * args.ld1 + col) = pack_bf16x4(ga_l);
      }
    }
  }
  // each row's sum over its 8 lanes (fixed butterfly order); lane q == 0 of the group writes
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float s = dgacc[i];
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    const int r = 4 * i + sub;
    if (q == 0 && r < nvalid) reinterpret_cast<float*>(args.out4)[(row0 + r) * args.ld2 + n] = s;
  }
}

// Gathering role of the ring forward (the pull dispatch): each of the first comm_ctas CTAs moves
// its share of each minibatch's rows (row i of the minibatch goes to CTA i % comm_ctas) from the
// token matrix into the minibatch's ring slot.  One SM moves rows on two paths at once, each of
// them bound by the latency of its copies in flight: warp 0 stages rows through shared memory
// with bulk async copies (lane 0 issues them, up to `ns` rows in flight; a row's staging buffer is
// refilled as soon as the store of the row before it has left it; the warp reads the rows' token
// indices 32 at a time, one window ahead), and the other warps copy rows through registers, one
// row per warp at a time, 16 bytes per lane and load.  Of every GATHER_PERIOD consecutive rows of
// the CTA, the first GATHER_BULK take the bulk path.  When the CTA's rows of a minibatch are in
// the ring it publishes their count.  A ring slot is overwritten only after every GEMM tile of the
// minibatch that held it has finished.
constexpr int GATHER_PERIOD = 9;
constexpr int GATHER_BULK = 4;

__device__ __forceinline__ void copy_row_warp(const uint4* __restrict__ src, uint4* __restrict__ dst, int vec,
                                              int lane) {
  constexpr int U = 16;
  for (int c = lane; c < vec; c += 32 * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c + u * 32 < vec) v[u] = __ldg(src + c + u * 32);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c + u * 32 < vec) dst[c + u * 32] = v[u];
  }
}

// Minibatch 0 of the ring, copied by every CTA of the launch before it takes its role (one row
// per warp at a time, rows dealt over all warps of the grid), so that no GEMM CTA waits for the
// gathering CTAs alone to fill the first slot: at T = 16384 with 2368-token minibatches the first
// slot holds 271 MB, about half a millisecond for 12 gathering SMs.  The gathering CTAs go on from
// minibatch 1.
__device__ inline void ring_gather_first(const GemmArgs& a) {
  const int warps = (int)(blockDim.x >> 5);
  const int gw = (int)blockIdx.x * warps + (int)(threadIdx.x >> 5);
  const int nw = (int)gridDim.x * warps;
  const int rows = min(a.mb_rows, a.R);
  const int slot = a.ring_shift % a.ring_slots;
  const int vec = a.H / 8;  // 16-byte words of a row
  int cnt = 0;
  for (int i = gw; i < rows; i += nw, ++cnt) {
    const int tok = a.src_of[i] / a.k_top;
    copy_row_warp(reinterpret_cast<const uint4*>(a.x + (size_t)tok * a.H),
                  reinterpret_cast<uint4*>(a.ring + ((size_t)slot * a.mb_rows + i) * a.H), vec, threadIdx.x & 31);
  }
  __threadfence();
  __syncwarp();
  if ((threadIdx.x & 31) == 0 && cnt > 0) atomicAdd(&a.gathered[0], cnt);
}

// staging barriers of ring_gather (one per row buffer of the CTA's shared memory, at most 16)
__device__ __forceinline__ int ring_gather_slots(const GemmArgs& a, int buf_bytes) {
  return min(16, buf_bytes / (a.H * 2));
}

// After ring_gather: its staging barriers are invalidated so that the CTA can set up other
// barriers in the same shared memory (every copy that completes on them has landed).
__device__ inline void ring_gather_retire(const GemmArgs& a, int buf_bytes, uint64_t* bars) {
  __syncthreads();
  if (threadIdx.x == 0)
    for (int j = 0; j < ring_gather_slots(a, buf_bytes); ++j)
      mbar_inval(smem_u32(&bars[j]));
  __syncthreads();
}

__device__ inline void ring_gather(const GemmArgs& a, uint8_t* buf, int buf_bytes, uint64_t* bars) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int copy_warps = (int)(blockDim.x >> 5) - 1;  // warps 1.. copy through registers
  const uint32_t row_bytes = (uint32_t)a.H * 2;
  const int ns = ring_gather_slots(a, buf_bytes);
  if (threadIdx.x == 0) {
    for (int j = 0; j < ns; ++j) mbar_init(smem_u32(&bars[j]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  volatile int no_abort = 0;
  long long gcount = 0;  // bulk rows this CTA has staged so far (slot = gcount % ns, parity = gcount / ns)
  long long issued = 0;  // bulk rows whose load has been issued
  for (int mb = 1; mb < a.n_mb; ++mb) {  // minibatch 0: ring_gather_first, by every CTA
    const int slot = (mb + a.ring_shift) % a.ring_slots;
    const int r0 = mb * a.mb_rows;
    const int rows = min(a.mb_rows, a.R - r0);
    int ok = 1;
    if (mb >= a.ring_slots && threadIdx.x == 0) {
      const int old = mb - a.ring_slots;
      ok = wait_counter(&a.consumed[old], a.consume_per_tile * (a.mb_start[old + 1] - a.mb_start[old]), a.status,
                        SITE_RING_WAIT);
    }
    if (__syncthreads_or(!ok)) return;
    const int cnt = rows > (int)blockIdx.x ? (rows - (int)blockIdx.x + a.comm_ctas - 1) / a.comm_ctas : 0;
    const int full = cnt / GATHER_PERIOD, rest = cnt % GATHER_PERIOD;
    const int n_bulk = full * GATHER_BULK + min(rest, GATHER_BULK);
    // the minibatch row of this CTA's q-th bulk / q-th register-copied row
    auto bulk_row = [&](int q) {
      return (int)blockIdx.x + ((q / GATHER_BULK) * GATHER_PERIOD + q % GATHER_BULK) * a.comm_ctas;
    };
    auto copy_row = [&](int q) {
      constexpr int NC = GATHER_PERIOD - GATHER_BULK;
      return (int)blockIdx.x + ((q / NC) * GATHER_PERIOD + GATHER_BULK + q % NC) * a.comm_ctas;
    };
    bool fail = false;
    if (warp == 0) {
      // token of the q-th bulk row: lane l holds rows base + l (cur) and base + 32 + l (nxt); q
      // only grows within a minibatch
      auto load_tok = [&](int q) {
        const int qq = q + lane;
        return qq < n_bulk ? a.src_of[r0 + bulk_row(qq)] / a.k_top : 0;
      };
      int base = 0;
      int cur = load_tok(0), nxt = load_tok(32);
      auto tok_at = [&](int q) {
        while (q >= base + 32) {
          base += 32;
          cur = nxt;
          nxt = load_tok(base + 32);
        }
        return __shfl_sync(0xffffffffu, cur, q - base);
      };
      auto issue_load = [&](long long g, int q) {
        const int tok = tok_at(q);
        if (lane == 0) {
          const int j = (int)(g % ns);
          mbar_arrive_expect_tx(smem_u32(&bars[j]), row_bytes);
          bulk_load_g2s(smem_u32(buf + (size_t)j * row_bytes), a.x + (size_t)tok * a.H, row_bytes,
                        smem_u32(&bars[j]));
        }
        issued = g + 1;
      };
      for (int q = 0; q < n_bulk && q < ns; ++q) issue_load(gcount + q, q);
      for (int q = 0; q < n_bulk; ++q) {
        const long long g = gcount + q;
        const int j = (int)(g % ns);
        int w_ok = 1;
        if (lane == 0) {
          w_ok = mbar_wait(smem_u32(&bars[j]), (uint32_t)((g / ns) & 1), &no_abort, a.status, SITE_RING_WAIT);
          if (w_ok) {
            bulk_store_s2g(a.ring + ((size_t)slot * a.mb_rows + bulk_row(q)) * a.H,
                           smem_u32(buf + (size_t)j * row_bytes), row_bytes);
            bulk_commit_group();
          }
        }
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          if (lane == 0) {
            // gave up: let the copies in flight land before the CTA leaves (bounded waits)
            bulk_wait_group_all();
            for (long long r = g; r < issued; ++r)
              mbar_wait(smem_u32(&bars[r % ns]), (uint32_t)((r / ns) & 1), &no_abort, a.status, SITE_RING_WAIT,
                        1000000ull);
          }
          fail = true;
          break;
        }
        // the staging buffer of row q-1 takes row q-1+ns once that row's store has read it
        if (q >= 1 && q - 1 + ns < n_bulk) {
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
          issue_load(g - 1 + ns, q - 1 + ns);
        }
      }
      gcount += n_bulk;
      if (!fail && lane == 0) {
        bulk_wait_group_all();  // the bulk rows are in the ring
        fence_proxy_async_global();
      }
      __syncwarp();
    } else {
      const int vec = a.H / 8;  // 16-byte words of a row
      for (int q = warp - 1; q < cnt - n_bulk; q += copy_warps) {
        const int i = copy_row(q);
        const int tok = a.src_of[r0 + i] / a.k_top;
        copy_row_warp(reinterpret_cast<const uint4*>(a.x + (size_t)tok * a.H),
                      reinterpret_cast<uint4*>(a.ring + ((size_t)slot * a.mb_rows + i) * a.H), vec, lane);
      }
      __threadfence();
    }
    if (__syncthreads_or(fail)) return;
    if (threadIdx.x == 0) {
      // every row of this CTA's share is in the ring: publish the count
      __threadfence();
      if (cnt > 0) atomicAdd(&a.gathered[mb], cnt);
    }
  }
}

template <int MODE, int EPI, int SPLIT, int BN_>
__global__ void __launch_bounds__(GemmCfg<MODE, EPI, SPLIT, BN_>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmO1,
                const __grid_constant__ CUtensorMap tmO2, const GemmArgs args) {
  using C = GemmCfg<MODE, EPI, SPLIT, BN_>;
  constexpr int BN = C::BN;
  constexpr int STAGES = C::STAGES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + C::RINGS_BYTES;               // epilogue output staging (C::STG_BYTES)
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::STG_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(staging + C::STG_BYTES + 256);
  int* s_toff = s_off + (args.E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + 2 + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * STAGES + 4]);

  if (MODE == MODE_RING) ring_gather_first(args);
  if (MODE == MODE_RING && (int)blockIdx.x < args.comm_ctas) {
    ring_gather(args, smem, STAGES * STAGE_BYTES, bars);
    return;
  }
  // the GEMM CTAs of this launch (all of them, except the gathering ones of MODE_RING)
  const int cta0 = (MODE == MODE_RING) ? (int)blockIdx.x - args.comm_ctas : (int)blockIdx.x;
  const int ncta = (MODE == MODE_RING) ? (int)gridDim.x - args.comm_ctas : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (MODE != MODE_DENSE && MODE != MODE_RING) {
    for (int i = threadIdx.x; i <= args.E; i += blockDim.x) {
      s_off[i] = args.offsets[i];
      s_toff[i] = (MODE == MODE_WGRAD) ? 0 : args.tile_off[i];
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int NT = C::n_tiles(args);
  const int total = (MODE == MODE_RING)       ? args.mb_start[args.n_mb]
                    : args.total_tiles >= 0 ? args.total_tiles
                                            : s_toff[args.E] * NT;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if (SPLIT == SPLIT_A) tma_prefetch_desc(&tmA2);
      if (SPLIT == SPLIT_B) tma_prefetch_desc(&tmB2);
      const uint64_t pol_act = l2_policy_evict_last();
      const uint64_t pol_once = l2_policy_evict_first();
      const uint64_t pol_shared = l2_policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      int ring_ready = -1;  // MODE_RING: last minibatch known to be gathered
      for (int g = cta0; g < total && ok; g += ncta) {
        const TileInfo t = decode_tile<MODE, EPI, SPLIT, BN_>(args, g, s_off, s_toff);
        // a weight tile is read once when its expert has a single m-tile; otherwise the
        // neighbouring CTAs that run the expert's other m-tiles read it again from L2
        const uint64_t pol_w = (MODE == MODE_WGRAD) ? pol_act : (t.mt > 1 ? pol_shared : pol_once);
        int a_row = t.row0;
        if (MODE == MODE_RING) {
          // rows of this minibatch must be in the ring before the first load of its tiles
          if (t.mb > ring_ready) {
            const int rows_mb = min(args.mb_rows, args.R - t.mb * args.mb_rows);
            if (!wait_counter(&args.gathered[t.mb], rows_mb, args.status, SITE_RING_WAIT)) {
              *abort_flag = 1;
              ok = false;
              break;
            }
            fence_proxy_async_global();
            ring_ready = t.mb;
          }
          a_row = ((t.mb + args.ring_shift) % args.ring_slots) * args.mb_rows + t.row0;
        }
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY,
                         kWaitLimitNs, 32)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sa2 = sa + A_TILE;                 // A lo (SPLIT_A)
          const uint32_t sb = sa + A_TILE * C::A_TILES;
          const uint32_t sb2 = sb + C::B_TILE;              // B lo (SPLIT_B)
          mbar_arrive_expect_tx(fb, C::TX_BYTES);
          const int k0 = kb * BK;
          if (MODE == MODE_DENSE) {
            tma_load_2d(sa, &tmA, fb, k0, t.row0, pol_act);
            tma_load_2d(sb, &tmB, fb, k0, t.n * BN, pol_w);
          } else if (MODE == MODE_ROWS || MODE == MODE_RING) {
            tma_load_2d(sa, &tmA, fb, k0, a_row, pol_act);
            if (SPLIT == SPLIT_A) tma_load_2d(sa2, &tmA2, fb, k0, a_row, pol_act);
            if (EPI == EPI_SWIGLU) {
              tma_load_3d(sb, &tmB, fb, k0, t.n * 128, t.e, pol_w);
              tma_load_3d(sb + C::B_TILE / 2, &tmB, fb, k0, args.I + t.n * 128, t.e, pol_w);
            } else {
              tma_load_3d(sb, &tmB, fb, k0, t.n * BN, t.e, pol_w);
            }
          } else if (MODE == MODE_DGRAD) {
            tma_load_2d(sa, &tmA, fb, k0, t.row0, pol_act);
            if (SPLIT == SPLIT_A) tma_load_2d(sa2, &tmA2, fb, k0, t.row0, pol_act);
#pragma unroll
            for (int q = 0; q < BN / 64; ++q)
              tma_load_3d(sb + q * MN_ATOM_BYTES, &tmB, fb, t.n * BN + q * 64, k0, t.e, pol_w);
          } else {  // WGRAD
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              tma_load_2d(sa + q * MN_ATOM_BYTES, &tmA, fb, t.m * BM + q * 64, t.row0 + k0, pol_act);
              if (SPLIT == SPLIT_A)
                tma_load_2d(sa2 + q * MN_ATOM_BYTES, &tmA2, fb, t.m * BM + q * 64, t.row0 + k0, pol_act);
            }
#pragma unroll
            for (int q = 0; q < BN / 64; ++q) {
              tma_load_2d(sb + q * MN_ATOM_BYTES, &tmB, fb, t.n * BN + q * 64, t.row0 + k0, pol_act);
              if (SPLIT == SPLIT_B)
                tma_load_2d(sb2 + q * MN_ATOM_BYTES, &tmB2, fb, t.n * BN + q * 64, t.row0 + k0, pol_act);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // Aborted: let the copies already in flight land before the CTA exits.
        const int outstanding = min(issued, STAGES);
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < outstanding; ++i) {
          if (--s < 0) {
            s = STAGES - 1;
            ph ^= 1;
          }
          volatile int no_abort = 0;
          mbar_wait(full_bar(s), ph, &no_abort, args.status, SITE_GEMM_DRAIN);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    bool any_mma = false;
    for (int g = cta0; g < total && ok; g += ncta) {
      const TileInfo t = decode_tile<MODE, EPI, SPLIT, BN_>(args, g, s_off, s_toff);
      if (t.nkb == 0) continue;
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait(tempty_bar(acc), acc_phase ^ 1, abort_flag, args.status, SITE_GEMM_MMA_TMEM_EMPTY);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * C::ACC_COLS;
      for (int kb = 0; kb < t.nkb; ++kb) {
        int f_ok = 1;
        if (lane == 0) f_ok = mbar_wait(full_bar(stage), phase, abort_flag, args.status, SITE_GEMM_MMA_FULL);
        if (!__shfl_sync(0xffffffffu, f_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* sa_ptr = smem + stage * STAGE_BYTES;
        const uint32_t sa = smem_u32(sa_ptr);
        const uint32_t sa2 = sa + A_TILE;
        const uint32_t sb = sa + A_TILE * C::A_TILES;
        const uint32_t sb2 = sb + C::B_TILE;
        int kvalid = BK;
        if (MODE == MODE_WGRAD) {
          kvalid = min(BK, t.rows - kb * BK);
          const int kend = (kvalid + 15) & ~15;
          if (kvalid < kend) {
            // zero the K rows [kvalid, kend) of every MN-major atom column of the stage
            constexpr int ATOMS = STAGE_BYTES / MN_ATOM_BYTES;
            const int nl = kend - kvalid;
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int idx = lane; idx < nl * ATOMS * 8; idx += 32) {
              const int chunk = idx & 7;
              const int li = idx >> 3;
              const int atom = li / nl;
              const int line = kvalid + (li - atom * nl);
              *reinterpret_cast<uint4*>(sa_ptr + atom * MN_ATOM_BYTES + line * 128 + chunk * 16) = z;
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (lane == 0) {
          const int nk16 = (kvalid + 15) >> 4;
          for (int k16 = 0; k16 < nk16; ++k16) {
            const uint32_t a_off = C::kAmn ? k16 * 2048 : k16 * 32;
            const uint32_t b_off = C::kBmn ? k16 * 2048 : k16 * 32;
            const uint32_t a_lbo = C::kAmn ? MOK_MN_LBO : 16, a_sbo = C::kAmn ? MOK_MN_SBO : 1024;
            const uint32_t b_lbo = C::kBmn ? MOK_MN_LBO : 16, b_sbo = C::kBmn ? MOK_MN_SBO : 1024;
            const uint64_t adesc = smem_desc_sw128(sa + a_off, a_lbo, a_sbo);
            const uint64_t bdesc = smem_desc_sw128(sb + b_off, b_lbo, b_sbo);
            umma_f16(d_tmem, adesc, bdesc, C::IDESC, (kb | k16) != 0 ? 1u : 0u);
            if (SPLIT == SPLIT_A) umma_f16(d_tmem, smem_desc_sw128(sa2 + a_off, a_lbo, a_sbo), bdesc, C::IDESC, 1u);
            if (SPLIT == SPLIT_B) umma_f16(d_tmem, adesc, smem_desc_sw128(sb2 + b_off, b_lbo, b_sbo), C::IDESC, 1u);
          }
          umma_commit(empty_bar(stage));
        }
        any_mma = true;
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(tfull_bar(acc));
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    // Wait for every MMA this CTA issued before TMEM is released.
    if (any_mma) {
      if (lane == 0) {
        umma_commit(drain_bar);
        volatile int no_abort = 0;
        mbar_wait(drain_bar, 0, &no_abort, args.status, SITE_GEMM_DRAIN);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 are reachable by this warp
    const int r_local = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int g = cta0; g < total; g += ncta) {
      const TileInfo t = decode_tile<MODE, EPI, SPLIT, BN_>(args, g, s_off, s_toff);
      if (MODE == MODE_WGRAD && t.nkb == 0) {
        // an expert without rows: its weight gradient is zero (transposed layout out[e][n][m])
        const size_t base = (size_t)t.e * args.M * args.N + (size_t)(t.n * BN) * args.M + t.m * BM + r_local;
        if (EPI == EPI_T_F32) {
          float* out = reinterpret_cast<float*>(args.out0) + base;
          for (int j = 0; j < BN; ++j) out[(size_t)j * args.M] = 0.0f;
        } else {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out0) + base;
          for (int j = 0; j < BN; ++j) out[(size_t)j * args.M] = __float2bfloat16_rn(0.0f);
        }
        continue;
      }
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.status, SITE_GEMM_EPI_TMEM_FULL, kWaitLimitNs,
                         256);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + acc * C::ACC_COLS + (uint32_t(quarter * 32) << 16);
      const bool valid = (MODE == MODE_WGRAD) ? true : (r_local < t.rows);
      const long long row = (MODE == MODE_WGRAD)  ? 0
                            : (MODE == MODE_RING) ? (long long)t.mb * args.mb_rows + t.row0 + r_local
                                                  : (long long)(t.row0 + r_local);

      const int nvalid = max(0, min(32, t.rows - quarter * 32));  // valid rows of this warp (ROWS / DGRAD)
      if (EPI == EPI_F32 && C::kTmaEpi) {
        epi_f32_tma<BN>(tacc, (long long)t.row0 + quarter * 32, nvalid, t.n, args, &tmO,
                        staging + (warp - 2) * 4096, lane);
      } else if (EPI == EPI_F32) {
        epi_f32_row<BN>(tacc, valid, row, t.n, args);
      } else if (EPI == EPI_SWIGLU && C::kTmaEpi) {
        epi_swiglu_tma<false>(tacc, (long long)t.row0 + quarter * 32, nvalid, t.n, args, &tmO, &tmO1, &tmO2,
                              staging + (warp - 2) * 4096, lane);
      } else if (EPI == EPI_T_F32 || EPI == EPI_T_BF16) {
        // out[e][n][m]: this warp's BN/32 blocks of 32 (m) x 32 (n).  All TMEM loads are issued
        // before one wait; each block goes to its own shared-memory buffer (m contiguous, lane =
        // m: conflict-free) and leaves through one TMA bulk tensor store.
        constexpr int NC = BN / 32;
        uint8_t* stg = staging + (warp - 2) * (NC * 4096);
        uint32_t v[NC][32];
#pragma unroll
        for (int c = 0; c < NC; ++c) tmem_ld_32x32b_x32(tacc + c * 32, v[c]);
        tmem_wait_ld();
        if (lane == 0) bulk_wait_group_read<0>();  // the previous tile's stores have read their buffers
        __syncwarp();
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          if (EPI == EPI_T_F32) {
            float* sb = reinterpret_cast<float*>(stg + c * 4096);
#pragma unroll
            for (int j = 0; j < 32; ++j) sb[j * 32 + lane] = __uint_as_float(v[c][j]);
          } else {
            __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stg + c * 4096);
#pragma unroll
            for (int j = 0; j < 32; ++j) sb[j * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[c][j]));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int c = 0; c < NC; ++c)
            tma_store_3d(&tmO, smem_u32(stg + c * 4096), t.m * BM + quarter * 32, t.n * BN + c * 32, t.e);
          bulk_commit_group();
        }
      } else if (EPI == EPI_SWIGLU) {
        epi_swiglu_row(tacc, valid, row, t.n, args);
      } else {  // EPI_SWIGLU_BWD
        epi_swiglu_bwd_cols<BN>(tacc, (long long)t.row0 + quarter * 32, nvalid, t.n, args, staging + (warp - 2) * 4096,
                                lane);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (MODE == MODE_RING && lane == 0) {
        // this warp is done with the tile: its minibatch's ring slot may be refilled once
        // every epilogue warp of every tile of the minibatch has counted in
        __threadfence();
        atomicAdd(&args.consumed[t.mb], 1);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    // TMA stores of this warp must finish reading shared memory (and land) before exit
    if ((MODE == MODE_WGRAD || C::kTmaEpi) && lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace mok
