// Block-scaled MXFP8 grouped GEMM on the FP8 tensor path (sm_103a): out[r][j] = sum_k X[r][k] W[e][j][k]
// over the expert-sorted rows r of each expert e, with X and W[e] in E4M3 and one E8M0 scale per
// 32 K-elements of each row, computed transposed, D[j][r] = W[e] X^T, by tcgen05.mma
// kind::mxf8f6f4 with scale_vec::1X: the tensor cores apply the scales themselves, so the E4M3
// bytes go from HBM to shared memory to the tensor cores unconverted.
//
// Shapes.  A CTA tile is 128 weight rows (the MMA's M) against one chunk of an expert's rows (its
// N, rounded up to 16, at most NMAX; the chunks of an expert start on 32-row boundaries of the
// padded row space of mx_tiles.h).  Each 128-byte K stage brings the weight tile(s), the chunk's
// rows and their scale blocks; the MMA warp copies the scales into TMEM (tcgen05.cp 32x128b.warpx4,
// one scale slot per stage) and issues four K = 32 MMAs, each picking its K-block's byte of the
// scale words.
//
//   MXE_SWIGLU  GEMM1 x_g W13[e]^T (K = H): two weight tiles per CTA tile, 128 gate rows and the
//               128 up rows of the same intermediate indices, two MMAs per K step sharing the rows;
//               h accumulates in TMEM columns [0, N), u in [256, 256 + N) of the same lanes.  The
//               epilogue stores h | u (fp32, for the backward) and a = silu(h) u quantised to MXFP8
//               along I: a warp's 32 lanes are 32 consecutive intermediate indices, i.e. one MX
//               block per row, whose maximum is a 5-step butterfly over the warp.  One accumulator.
//   MXE_F32     GEMM2 a W2[e]^T (K = I): one weight tile per CTA tile, fp32 output; two
//               accumulators, so the epilogue of a tile overlaps the main loop of the next.
//
// Roles: warp 0 TMA producer, warp 1 MMA issuer (one elected thread), warps 2..5 epilogue (warp w
// reads TMEM lane quarter w % 4).  Tiles (expert e, weight tile m, row chunk c; c fastest, then m)
// are dealt round-robin in a fixed order; every output element is one tile's accumulator, reduced
// over K in a fixed order, so the results are deterministic.  Every wait is bounded.
#pragma once
#include <cuda_bf16.h>

#include "mx.cuh"
#include "mx_tiles.h"
#include "ptx.cuh"

namespace mok {

enum MxEpi { MXE_SWIGLU = 0, MXE_F32 = 1 };

struct MxGemmArgs {
  int E;
  int K;                  // reduction length, a multiple of 128
  int Nw;                 // rows of each expert's weight matrix (2I for GEMM1, H for GEMM2)
  int MT;                 // CTA weight tiles per expert (GEMM1: I / 128 gate-up pairs, GEMM2: H / 128)
  int I;                  // GEMM1: intermediate width
  int G;                  // row groups of the row operand's scale blocks (mx_row_groups)
  const int* offsets;     // [E+1] expert row offsets (schedule order)
  const int* blk_off;     // [E+1] 32-row blocks before each expert (padded row space)
  const uint8_t* w_sf;    // [E][Nw/128][K/128][512] weight scale blocks
  const uint8_t* x_sf;    // [G][K/128][512] row scale blocks
  float* out;             // GEMM1: h | u [R][2I]; GEMM2: o [R][Nw]
  long long ld;           // row stride of out (elements)
  uint8_t* aq;            // GEMM1: a, E4M3 [padded rows][I]
  uint8_t* asf;           // GEMM1: its scale blocks [G][I/128][512]
  int* status;
};

template <int EPI, int NMAX_, int STAGES_>
struct MxCfg {
  static constexpr bool kPaired = EPI == MXE_SWIGLU;
  static constexpr int NMAX = NMAX_;
  static constexpr int STAGES = STAGES_;
  static constexpr int NA = kPaired ? 2 : 1;                 // weight tiles per CTA tile
  static constexpr int ACCS = kPaired ? 1 : 2;               // accumulators
  static constexpr int A_TILE = 128 * MX_BK;                 // 16 KB per weight tile and stage
  static constexpr int B_BYTES = NMAX * MX_BK;
  static constexpr int NSFB = (NMAX + 127) / 128;            // row scale blocks per stage
  static constexpr int SF_OFF = NA * A_TILE + B_BYTES;       // scale blocks after the operands
  static constexpr int STAGE_BYTES = (SF_OFF + (NA + NSFB) * MX_SF_BLOCK + 1023) & ~1023;
  // TMEM: the accumulator(s), then one scale slot per stage (4 columns per scale block)
  static constexpr int ACC_STRIDE = kPaired ? 256 : NMAX;    // paired: up rows at column 256
  static constexpr int SF_BASE = kPaired ? NMAX : 2 * NMAX;
  static constexpr int SLOT_COLS = 4 * (NA + NSFB);
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 192;
  static_assert(NMAX % 32 == 0 && NMAX >= 32 && NMAX <= 256, "chunk rows");
  static_assert(kPaired ? (SF_BASE + STAGES * SLOT_COLS <= 256) : (SF_BASE + STAGES * SLOT_COLS <= TMEM_COLS),
                "scale slots must fit beside the accumulators");
  static __host__ __device__ constexpr size_t smem_bytes(int E) {
    return size_t(STAGES) * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/ + size_t(3) * (E + 1) * 4;
  }
};

// 32 lanes' maximum (every lane gets it); a max is exact in any order.
__device__ __forceinline__ float warp_max32(float v) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, s));
  return v;
}

// Scale byte of padded row p, 32-block kb of K stage s, into the four row-group blocks that hold
// it (blocks [G][S][512], S stages).
__device__ __forceinline__ void mx_store_row_scale(uint8_t* sf, int S, int p, int s, int kb, uint8_t v) {
  const int g_top = p >> 5;
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int g = g_top - jj;
    if (g >= 0) sf[((size_t)g * S + s) * MX_SF_BLOCK + (p & 31) * 16 + jj * 4 + (kb & 3)] = v;
  }
}

// tmW: the expert weights as a 2-D E4M3 tensor [E * Nw][K], 128 x 128-byte boxes.  tmX: the padded
// row operand [rows][K], 32-row x 128-byte boxes.
template <int EPI, int NMAX, int STAGES>
__global__ void __launch_bounds__(192, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const MxGemmArgs args) {
  using C = MxCfg<EPI, NMAX, STAGES>;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + 256);
  int* s_boff = s_off + (args.E + 1);
  int* s_coff = s_boff + (args.E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + 2 + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * STAGES + 4]);

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
  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) {
    s_off[i] = args.offsets[i];
    s_boff[i] = args.blk_off[i];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < args.E; ++e) {
      s_coff[e] = acc;
      acc += (s_off[e + 1] - s_off[e] + C::NMAX - 1) / C::NMAX;
    }
    s_coff[args.E] = acc;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int MT = args.MT;
  const int total = s_coff[args.E] * MT;
  const int nkb = args.K / MX_BK;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      const uint64_t pol_rows = l2_policy_evict_last();   // rows: read by every weight tile
      const uint64_t pol_once = l2_policy_evict_first();  // a weight tile read by one chunk
      const uint64_t pol_shared = l2_policy_evict_normal();
      const int wtiles = args.Nw / 128;
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int g = blockIdx.x; g < total && ok; g += gridDim.x) {
        const MxTile t = decode_mx_tile(g, MT, args.E, C::NMAX, s_off, s_boff, s_coff);
        const int nsfb = (t.nload + 127) / 128;
        const uint32_t tx = C::NA * C::A_TILE + t.nload * MX_BK + (C::NA + nsfb) * MX_SF_BLOCK;
        const uint64_t pol_w = t.nc > 1 ? pol_shared : pol_once;
        int wt[2];  // weight tiles (128-row units of the expert's matrix) of this CTA tile
        if (EPI == MXE_SWIGLU) {
          wt[0] = t.m;                 // gate rows 128 m ..
          wt[1] = args.I / 128 + t.m;  // up rows I + 128 m ..
        } else {
          wt[0] = wt[1] = t.m;
        }
        const int g0 = t.prow0 >> 5;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY,
                         kWaitLimitNs, 32)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, tx);
          const int k0 = kb * MX_BK;
#pragma unroll
          for (int a = 0; a < C::NA; ++a) {
            tma_load_2d(smem_u32(sa + a * C::A_TILE), &tmW, fb, k0, t.e * args.Nw + wt[a] * 128, pol_w);
            const uint8_t* sf = args.w_sf + (((size_t)t.e * wtiles + wt[a]) * nkb + kb) * MX_SF_BLOCK;
            bulk_load_g2s(smem_u32(sa + C::SF_OFF + a * MX_SF_BLOCK), sf, MX_SF_BLOCK, fb);
          }
          uint8_t* sb = sa + C::NA * C::A_TILE;
          for (int r = 0; r < t.nload; r += 32) tma_load_2d(smem_u32(sb + r * MX_BK), &tmX, fb, k0, t.prow0 + r, pol_rows);
          for (int b = 0; b < nsfb; ++b) {
            const uint8_t* sf = args.x_sf + ((size_t)(g0 + 4 * b) * nkb + kb) * MX_SF_BLOCK;
            bulk_load_g2s(smem_u32(sa + C::SF_OFF + (C::NA + b) * MX_SF_BLOCK), sf, MX_SF_BLOCK, fb);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // Aborted: wait for the stages armed last so that no copy is still landing at exit.
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
    for (int g = blockIdx.x; g < total && ok; g += gridDim.x) {
      const MxTile t = decode_mx_tile(g, MT, args.E, C::NMAX, s_off, s_boff, s_coff);
      const int nsfb = (t.nload + 127) / 128;
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(tempty_bar(acc), acc_phase ^ 1, abort_flag, args.status, SITE_GEMM_MMA_TMEM_EMPTY);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * C::ACC_STRIDE;
      for (int kb = 0; kb < nkb; ++kb) {
        int f_ok = 1;
        if (lane == 0) f_ok = mbar_wait(full_bar(stage), phase, abort_flag, args.status, SITE_GEMM_MMA_FULL);
        if (!__shfl_sync(0xffffffffu, f_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint8_t* sa = smem + stage * STAGE_BYTES;
          const uint32_t sf_col = tmem_base + C::SF_BASE + stage * C::SLOT_COLS;
          // this stage's scales into its TMEM slot (the slot's previous MMAs completed before the
          // producer refilled the stage); tcgen05.cp and the MMAs below run in issue order
#pragma unroll
          for (int a = 0; a < C::NA; ++a)
            tmem_cp_32x128b_warpx4(sf_col + 4 * a, smem_desc_noswizzle(smem_u32(sa + C::SF_OFF + a * MX_SF_BLOCK), 0, 128));
          for (int b = 0; b < nsfb; ++b)
            tmem_cp_32x128b_warpx4(sf_col + 4 * (C::NA + b),
                                   smem_desc_noswizzle(smem_u32(sa + C::SF_OFF + (C::NA + b) * MX_SF_BLOCK), 0, 128));
          const uint32_t sb = smem_u32(sa + C::NA * C::A_TILE);
#pragma unroll
          for (int k4 = 0; k4 < MX_BK / 32; ++k4) {
            const uint32_t idesc = idesc_mxf8_e4m3(128, t.n, k4, k4);
            const uint64_t bdesc = smem_desc_sw128(sb + k4 * 32, 16, 1024);
            const uint32_t accumulate = (kb | k4) != 0 ? 1u : 0u;
#pragma unroll
            for (int a = 0; a < C::NA; ++a) {
              const uint64_t adesc = smem_desc_sw128(smem_u32(sa + a * C::A_TILE) + k4 * 32, 16, 1024);
              umma_mxf8(d_tmem + a * 256, adesc, bdesc, idesc, sf_col + 4 * a, sf_col + 4 * C::NA, accumulate);
            }
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
      acc = (acc + 1) % C::ACCS;
      if (acc == 0) acc_phase ^= 1;
    }
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
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int g = blockIdx.x; g < total; g += gridDim.x) {
      const MxTile t = decode_mx_tile(g, MT, args.E, C::NMAX, s_off, s_boff, s_coff);
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.status, SITE_GEMM_EPI_TMEM_FULL, kWaitLimitNs,
                         256);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + acc * C::ACC_STRIDE + (uint32_t(quarter * 32) << 16);
      if (EPI == MXE_SWIGLU) {
        // this thread's intermediate index; h in column n, u in column 256 + n of its lane
        const int I = args.I;
        const int i = t.m * 128 + 32 * quarter + lane;
        float* hrow = args.out + (long long)t.row0 * args.ld + i;
        uint8_t* arow = args.aq + (long long)t.prow0 * I + i;
        const int S = I / MX_BK;
#pragma unroll 1
        for (int n0 = 0; n0 < t.nload; n0 += 8) {
          uint32_t hv[8], uv[8];
          tmem_ld_32x32b_x8(tacc + n0, hv);
          tmem_ld_32x32b_x8(tacc + 256 + n0, uv);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int n = n0 + j;
            const bool valid = n < t.rows;  // rows past the expert's end become zero rows of a
            const float h = valid ? __uint_as_float(hv[j]) : 0.0f;
            const float u = valid ? __uint_as_float(uv[j]) : 0.0f;
            if (valid) {
              hrow[(long long)n * args.ld] = h;
              hrow[(long long)n * args.ld + I] = u;
            }
            const float a = h / (1.0f + __expf(-h)) * u;
            // one MX block: this row's 32 intermediate indices of the warp
            const int X = mx_exponent(warp_max32(fabsf(a)));
            const uint16_t q = e4m3x2_from_f32(a * exp2_int(-X), 0.0f);
            arow[(long long)n * I] = (uint8_t)(q & 0xff);
            if (lane == 0) mx_store_row_scale(args.asf, S, t.prow0 + n, t.m, quarter, (uint8_t)(X + 127));
          }
        }
      } else {
        // this thread's output column; the accumulator's columns are the chunk's rows
        const int j = t.m * 128 + 32 * quarter + lane;
        float* o = args.out + (long long)t.row0 * args.ld + j;
#pragma unroll 1
        for (int c = 0; c * 32 < t.rows; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + c * 32, v);
          tmem_wait_ld();
          const int nr = min(32, t.rows - c * 32);
          float* oc = o + (long long)(c * 32) * args.ld;
          if (nr == 32) {
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) oc[(long long)ii * args.ld] = __uint_as_float(v[ii]);
          } else {
#pragma unroll
            for (int ii = 0; ii < 32; ++ii)
              if (ii < nr) oc[(long long)ii * args.ld] = __uint_as_float(v[ii]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      acc = (acc + 1) % C::ACCS;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace mok
