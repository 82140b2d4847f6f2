// Block-scaled MXFP8 grouped GEMM on CTA pairs (sm_103a): out[r][j] = sum_k X[r][k] W[e][j][k] over the
// expert-sorted rows r of each expert e, with X and W[e] in E4M3 and one E8M0 scale per 32 K-elements
// of each row, computed transposed, D[j][r] = W[e] X^T, by tcgen05.mma.cta_group::2 kind::mxf8f6f4
// with scale_vec::1X: the tensor cores apply the scales themselves, so the E4M3 bytes go from HBM to
// shared memory to the tensor cores unconverted.
//
// Shapes.  A pair tile is 256 weight rows (the MMA's M, 128 per CTA) against one chunk of an
// expert's rows (its N, a multiple of 16 up to NMAX, split by columns across the pair: each CTA
// stages N / 2 rows).  The chunks of an expert start on 32-row boundaries of the padded row space of
// mx_tiles.h.  Each 128-byte K stage brings, per CTA, its 128 weight rows, its half of the chunk's
// rows, the scale block of its weight rows and the scale blocks of all N rows; the even CTA copies
// the scales into both CTAs' TMEM (tcgen05.cp.cta_group::2: each CTA's shared memory into its own
// TMEM, one scale slot per stage) and issues four K = 32 MMAs, each picking its K-block's byte of
// the scale words.  Two accumulators: the epilogue of a tile overlaps the main loop of the next.
//
//   MXE_SWIGLU      GEMM1 x_g W13[e]^T (K = H).  Each CTA's 128 weight rows are 64 gate rows and the
//                   64 up rows of the same intermediate indices (a box of the [E][2][I][H] view), so h
//                   and u of one (row, i) sit on TMEM lane quarters q and q + 2; the gate warp hands h
//                   to the up warp through shared memory.  Out: h | u (fp32, for the backward) and
//                   a = silu(h) u quantised to MXFP8 along I: a warp's 32 lanes are 32 consecutive
//                   intermediate indices, one MX block per row, whose maximum is a butterfly.
//   MXE_F32         GEMM2 a W2[e]^T (K = I) and dX_g = dHU W13[e] (K = 2I): fp32 out.
//   MXE_SWIGLU_BWD  dA' = dY_g W2[e] (K = H, W2 stored transposed [I][H]).  Out: the SwiGLU backward
//                   dh = g dA' u silu'(h), du = g dA' silu(h) as bf16 hi / lo pairs and as MXFP8 along
//                   2I (the row operand of dX_g), and the partial gate gradient <dA', a> of the CTA's
//                   128 intermediate indices per row (a fixed-order reduction over lanes and warps).
//
// Roles (both CTAs): warp 0 TMA producer, warp 1 MMA issuer (even CTA, one elected thread), warps
// 2..5 epilogue (warp w reads TMEM lane quarter w % 4).  Barriers as in gemm_narrow.cuh: full[s] in
// the even CTA (one arrival with the bytes of both CTAs), empty[s] and tfull[a] in both CTAs
// (multicast commits), tempty[a] in the even CTA (8 arrivals).  Tiles (expert e, weight tile m, row
// chunk c; c fastest, then m) are dealt round-robin to the pairs in a fixed order; every output
// element is one tile's accumulator, reduced over K in a fixed order, so the results are
// deterministic.  Every wait is bounded.
#pragma once
#include <cuda_bf16.h>

#include "mx.cuh"
#include "mx_tiles.h"
#include "ptx.cuh"

namespace mok {

enum MxEpi { MXE_SWIGLU = 0, MXE_F32 = 1, MXE_SWIGLU_BWD = 2 };

struct MxGemmArgs {
  int E;
  int K;                  // reduction length, a multiple of 128
  int MT;                 // pair weight tiles per expert (GEMM1: I / 128; else ceil(Nw / 256))
  int Nw;                 // rows of each expert's weight matrix (a multiple of 128)
  int I;                  // intermediate width (SwiGLU epilogues)
  int N_out;              // F32: output columns (the weight rows of an expert)
  int sfa_tiles;          // 128-row scale tiles per expert of the weight matrix
  const int* offsets;     // [E+1] expert row offsets (schedule order)
  const int* blk_off;     // [E+1] 32-row blocks before each expert (padded row space)
  float* out;             // SWIGLU: h | u [R][2I]; F32: [R][ld]
  long long ld;           // row stride of out (elements)
  uint8_t* q;             // SWIGLU: a, E4M3 [padded rows][I]; BWD: dh | du, E4M3 [padded rows][2I]
  uint8_t* qsf;           // its scale blocks [G][width / 128][512]
  const float* hu;        // BWD: saved h | u [R][2I]
  const float* gate_row;  // BWD: gate of each row
  __nv_bfloat16* dhu_hi;  // BWD: dh | du hi [R][2I]
  __nv_bfloat16* dhu_lo;  // BWD: lo
  float* dg_part;         // BWD: partial gate gradients [R][I / 128]
  int* status;
};

template <int EPI, int NMAX_, int STAGES_>
struct MxCfg {
  static constexpr int NMAX = NMAX_;                         // rows of a chunk at most
  static constexpr int STAGES = STAGES_;
  static constexpr int A_TILE = 128 * MX_BK;                 // 16 KB: one CTA's weight rows per stage
  static constexpr int XROWS = ((NMAX / 2) + 31) & ~31;      // one CTA's rows per stage (32-row boxes)
  static constexpr int B_BYTES = XROWS * MX_BK;
  static constexpr int NSFB = (NMAX + 127) / 128;            // row scale blocks per stage
  static constexpr int SF_OFF = A_TILE + B_BYTES;            // scale blocks after the operands
  static constexpr int STAGE_BYTES = (SF_OFF + (1 + NSFB) * MX_SF_BLOCK + 1023) & ~1023;
  static constexpr int ACCS = 2;
  static constexpr int SF_BASE = ACCS * NMAX;                // TMEM: accumulators, then one scale slot per stage
  static constexpr int SLOT_COLS = 4 * (1 + NSFB);
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 192;
  // 32 x 32 fp32 blocks with rows XLD floats apart (16-byte aligned, conflict-free 16-byte row reads):
  // SwiGLU: one per pair of gate / up warps (h, then a in place); backward: one per epilogue warp
  static constexpr int XLD = 36;
  static constexpr int XBLK = 32 * XLD * 4;
  static constexpr int XBUF_BYTES = EPI == MXE_SWIGLU ? 2 * XBLK : EPI == MXE_SWIGLU_BWD ? 4 * XBLK : 0;
  static constexpr int DGBUF_BYTES = EPI == MXE_SWIGLU_BWD ? 4 * 32 * 4 : 0;      // per-warp gate partials
  static_assert(NMAX % 32 == 0 && NMAX >= 32 && NMAX <= 256, "chunk rows");
  static_assert(SF_BASE + STAGES * SLOT_COLS <= TMEM_COLS, "scale slots must fit beside the accumulators");
  static __host__ __device__ constexpr size_t smem_bytes(int E) {
    return size_t(STAGES) * STAGE_BYTES + XBUF_BYTES + DGBUF_BYTES + 1024 /*align*/ + 256 /*barriers*/ +
           size_t(3) * (E + 1) * 4;
  }
};

// 32 lanes' maximum (every lane gets it); a max is exact in any order.
__device__ __forceinline__ float warp_max32(float v) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, s));
  return v;
}

// Lane l receives sum over the warp's lanes of v[l] (each lane holds 32 values, one per column):
// recursive halving, each stage keeps half of the columns and adds the partner lane's half, a fixed
// order of additions per column (31 shuffles instead of 32 x 5).
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const float send = upper ? v[k] : v[k + w];
      const float keep = upper ? v[k + w] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
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

// One MX block held by one thread: the 32 consecutive elements of row p at blk[0..31] (shared
// memory, 16-byte aligned); the E4M3 bytes go to q (16-byte aligned, one 32-byte store) and the
// scale to its four row-group blocks (stage s, 32-block kb).
__device__ __forceinline__ void mx_quantize_row32(const float* blk, uint8_t* q, uint8_t* sf, int S, int p, int s,
                                                  int kb) {
  float v[32];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 f = reinterpret_cast<const float4*>(blk)[c];
    v[4 * c] = f.x;
    v[4 * c + 1] = f.y;
    v[4 * c + 2] = f.z;
    v[4 * c + 3] = f.w;
  }
  __align__(16) uint8_t bytes[32];
  const int X = mx_quantize32(v, bytes);
  uint4* dst = reinterpret_cast<uint4*>(q);
  dst[0] = *reinterpret_cast<const uint4*>(bytes);
  dst[1] = *reinterpret_cast<const uint4*>(bytes + 16);
  mx_store_row_scale(sf, S, p, s, kb, (uint8_t)(X + 127));
}

// tmW: the expert weights in E4M3 (SwiGLU: a 4-D view [E][2][I][H], boxes of 128 bytes x 64 rows x
// both halves; else [E * Nw][K], boxes of 128 bytes x 128 rows).  tmX: the padded row operand
// [rows][K], 32-row boxes.  tmWS / tmXS: scale blocks seen as [blocks][4][128] bytes, one block per box.
template <int EPI, int NMAX, int STAGES>
__global__ void __launch_bounds__(192, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmWS, const __grid_constant__ CUtensorMap tmXS,
                   const MxGemmArgs args) {
  using C = MxCfg<EPI, NMAX, STAGES>;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xbuf = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);                    // C::XBUF_BYTES
  float* dgbuf = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + C::XBUF_BYTES);   // C::DGBUF_BYTES
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + C::XBUF_BYTES + C::DGBUF_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + 256);
  int* s_boff = s_off + (args.E + 1);
  int* s_coff = s_boff + (args.E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
  const int pair = (int)blockIdx.x >> 1;
  const int npairs = (int)gridDim.x >> 1;
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
      mbar_init(tempty_bar(a), 8);
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
    tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int MT = args.MT;
  const int total = s_coff[args.E] * MT;
  const int nkb = args.K / MX_BK;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmWS);
      tma_prefetch_desc(&tmXS);
      const uint64_t pol_rows = l2_policy_evict_last();   // rows: read by every weight tile
      const uint64_t pol_once = l2_policy_evict_first();  // a weight tile read by one chunk
      const uint64_t pol_shared = l2_policy_evict_normal();
      const uint32_t full0_cl = mapa_shared(full_bar(0), 0);  // the even CTA's full barriers
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int g = pair; g < total && ok; g += npairs) {
        const MxTile t = decode_mx_tile(g, MT, args.E, C::NMAX, s_off, s_boff, s_coff);
        const int half = t.n >> 1;                          // rows of this CTA's half of N
        const int nbox = (half + 31) >> 5;                  // 32-row boxes (<= XROWS / 32)
        const int nsfb = (t.n + 127) >> 7;                  // scale blocks of all N rows
        const uint32_t pair_tx = 2u * (C::A_TILE + nbox * 32 * MX_BK + (1 + nsfb) * MX_SF_BLOCK);
        const uint64_t pol_w = t.nc > 1 ? pol_shared : pol_once;
        // this CTA's 128-row scale tile of the weight matrix (SwiGLU: its 64 gate + 64 up rows)
        const int wtile = 2 * t.m + (int)rank;
        const int g0 = t.prow0 >> 5;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait<true>(empty_bar(stage), phase ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY,
                               kWaitLimitNs, 32)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0_cl + 8u * stage;
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + C::A_TILE;
          const uint32_t ssf = sa + C::SF_OFF;
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), pair_tx);
          const int k0 = kb * MX_BK;
          if (EPI == MXE_SWIGLU) {
            // 64 gate rows, then the 64 up rows of the same intermediate indices
            tma_load_4d_pair(sa, &tmW, fb, k0, t.m * 128 + 64 * (int)rank, 0, t.e, pol_w);
          } else {
            tma_load_2d_pair(sa, &tmW, fb, k0, t.e * args.Nw + t.m * 256 + 128 * (int)rank, pol_w);
          }
          tma_load_3d_pair(ssf, &tmWS, fb, 0, 0, (t.e * args.sfa_tiles + wtile) * nkb + kb, pol_w);
          const int x_row = t.prow0 + (int)rank * half;
          for (int b = 0; b < nbox; ++b) tma_load_2d_pair(sb + b * 32 * MX_BK, &tmX, fb, k0, x_row + 32 * b, pol_rows);
          for (int b = 0; b < nsfb; ++b)
            tma_load_3d_pair(ssf + (1 + b) * MX_SF_BLOCK, &tmXS, fb, 0, 0, (g0 + 4 * b) * nkb + kb, pol_rows);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        if (rank == 0) {
          // Aborted: the even CTA's full barriers count both CTAs' bytes; wait for the stages
          // it armed so that no copy is still landing when the pair exits.
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
        } else {
          // the peer cannot observe its own copies: give those in flight time to land
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 100000ull) __nanosleep(1000);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool any_mma = false;
      for (int g = pair; g < total && ok; g += npairs) {
        const MxTile t = decode_mx_tile(g, MT, args.E, C::NMAX, s_off, s_boff, s_coff);
        const int nsfb = (t.n + 127) >> 7;
        int w_ok = 1;
        if (lane == 0)
          w_ok = mbar_wait<true>(tempty_bar(acc), acc_phase ^ 1, abort_flag, args.status, SITE_GEMM_MMA_TMEM_EMPTY);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::NMAX;
        for (int kb = 0; kb < nkb; ++kb) {
          int f_ok = 1;
          if (lane == 0) f_ok = mbar_wait<true>(full_bar(stage), phase, abort_flag, args.status, SITE_GEMM_MMA_FULL);
          if (!__shfl_sync(0xffffffffu, f_ok, 0)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t sb = sa + C::A_TILE;
            const uint32_t ssf = sa + C::SF_OFF;
            const uint32_t sf_col = tmem_base + C::SF_BASE + stage * C::SLOT_COLS;
            // this stage's scales into its TMEM slot of both CTAs (each CTA's own shared memory:
            // its weight rows' scales and all N rows' scales); the slot's previous MMAs completed
            // before the producer refilled the stage, and tcgen05.cp and the MMAs run in issue order
            tmem_cp_32x128b_warpx4_pair(sf_col, smem_desc_noswizzle(ssf, 0, 128));
            for (int b = 0; b < nsfb; ++b)
              tmem_cp_32x128b_warpx4_pair(sf_col + 4 * (1 + b), smem_desc_noswizzle(ssf + (1 + b) * MX_SF_BLOCK, 0, 128));
#pragma unroll
            for (int k4 = 0; k4 < MX_BK / 32; ++k4) {
              const uint64_t adesc = smem_desc_sw128(sa + k4 * 32, 16, 1024);
              const uint64_t bdesc = smem_desc_sw128(sb + k4 * 32, 16, 1024);
              umma_mxf8_pair(d_tmem, adesc, bdesc, idesc_mxf8_e4m3(256, t.n, k4, k4), sf_col, sf_col + 4,
                             (kb | k4) != 0 ? 1u : 0u);
            }
            umma_commit_pair(empty_bar(stage), 0x3);
          }
          any_mma = true;
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if (lane == 0) umma_commit_pair(tfull_bar(acc), 0x3);
        __syncwarp();
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (any_mma) {
        if (lane == 0) {
          umma_commit_pair(drain_bar, 0x1);
          volatile int no_abort = 0;
          mbar_wait(drain_bar, 0, &no_abort, args.status, SITE_GEMM_DRAIN);
        }
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 are reachable by this warp
    const uint32_t tempty0_cl = mapa_shared(tempty_bar(0), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int g = pair; g < total; g += npairs) {
      const MxTile t = decode_mx_tile(g, MT, args.E, C::NMAX, s_off, s_boff, s_coff);
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait<true>(tfull_bar(acc), acc_phase, abort_flag, args.status, SITE_GEMM_EPI_TMEM_FULL,
                               kWaitLimitNs, 256);
      const uint32_t tacc = tmem_base + acc * C::NMAX + (uint32_t(quarter * 32) << 16);
      if (EPI == MXE_SWIGLU) {
        // the two warps that share intermediate indices agree on stopping (one of them may have
        // given up waiting while the other saw the accumulator complete)
        const int qp = quarter & 1;
        const bool w_fail = !__shfl_sync(0xffffffffu, w_ok, 0);
        if (named_bar_any(1 + qp, 64, w_fail)) break;
        tc_fence_after();
        const bool gate = quarter < 2;  // lanes of gate rows (h); quarter + 2 holds u
        const int I = args.I;
        const int i = t.m * 128 + 64 * (int)rank + 32 * qp + lane;
        const int S = I / MX_BK;
        const int kb_a = 2 * (int)rank + qp;  // 32-block of i inside its 128-element stage t.m
        float* hu = args.out + (long long)t.row0 * args.ld;
        // [32 rows][32 indices]: h parked by the gate warp, then a = silu(h) u written in place by the
        // up warp, then each up-warp thread quantises one row (32 consecutive i: one MX block)
        float* xb = xbuf + qp * (C::XBLK / 4);
#pragma unroll 1
        for (int c = 0; c * 32 < t.nload; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + c * 32, v);
          tmem_wait_ld();
          const int nr = min(32, t.rows - c * 32);  // rows of the expert in this block (may be <= 0)
          float* hp = hu + (long long)(c * 32) * args.ld + (gate ? i : I + i);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nr) hp[(long long)j * args.ld] = __uint_as_float(v[j]);
          if (gate) {
#pragma unroll
            for (int j = 0; j < 32; ++j) xb[j * C::XLD + lane] = __uint_as_float(v[j]);
          }
          named_bar_sync(1 + qp, 64);  // h of this block is in shared memory
          if (!gate) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const bool valid = j < nr;  // rows past the expert's end become zero rows of a
              const float h = valid ? xb[j * C::XLD + lane] : 0.0f;
              const float u = valid ? __uint_as_float(v[j]) : 0.0f;
              xb[j * C::XLD + lane] = h / (1.0f + __expf(-h)) * u;
            }
            __syncwarp();
            const int p = t.prow0 + c * 32 + lane;
            mx_quantize_row32(xb + lane * C::XLD, args.q + (long long)p * I + (i - lane), args.qsf, S, p, t.m, kb_a);
          }
          named_bar_sync(1 + qp, 64);  // the up warp is done with the block
        }
      } else if (EPI == MXE_F32) {
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
        tc_fence_after();
        // this thread's output column; the accumulator's columns are the chunk's rows
        const int j = t.m * 256 + 128 * (int)rank + 32 * quarter + lane;
        const bool jv = j < args.N_out;
        float* o = args.out + (long long)t.row0 * args.ld + j;
#pragma unroll 1
        for (int c = 0; c * 32 < t.rows; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + c * 32, v);
          tmem_wait_ld();
          const int nr = min(32, t.rows - c * 32);
          if (jv) {
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
      } else {  // MXE_SWIGLU_BWD
        // the four epilogue warps of the CTA agree on stopping (they reduce the gate partials together)
        const bool w_fail = !__shfl_sync(0xffffffffu, w_ok, 0);
        if (named_bar_any(1, 128, w_fail)) break;
        tc_fence_after();
        const int I = args.I;
        const int twoI = 2 * I;
        // the pair tile reaches past I (a multiple of 128, not 256): this CTA's 128 indices lie
        // beyond it and it has nothing to store (the same for all four warps of the CTA)
        const bool cta_in = t.m * 256 + 128 * (int)rank < I;
        const int i = t.m * 256 + 128 * (int)rank + 32 * quarter + lane;  // this thread's intermediate index
        const int S = twoI / MX_BK;
        const int s_h = i >> 7, s_u = (I + i) >> 7;            // K stages of dX_g holding dh_i, du_i
        const int kb_h = (i >> 5) & 3, kb_u = ((I + i) >> 5) & 3;
        const int part = 2 * t.m + (int)rank;                   // this CTA's 128 intermediate indices
        const int nparts = I / 128;
#pragma unroll 1
        for (int c = 0; cta_in && c * 32 < t.nload; ++c) {
          const int nr = min(32, t.rows - c * 32);
          const int p0 = t.prow0 + c * 32;
          const long long r0 = (long long)t.row0 + c * 32;
          // the block's h | u and gates first, so that their latency overlaps the TMEM read
          float hv[32], uv[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            hv[j] = j < nr ? args.hu[(r0 + j) * twoI + i] : 0.0f;
            uv[j] = j < nr ? args.hu[(r0 + j) * twoI + I + i] : 0.0f;
          }
          const float g_lane = lane < nr ? args.gate_row[r0 + lane] : 0.0f;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + c * 32, v);
          tmem_wait_ld();
          float dgp[32];
          float* xb = xbuf + quarter * (C::XBLK / 4);  // [32 rows][32 indices] of this warp
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const bool valid = j < nr;
            const float h = hv[j], u = uv[j];
            const float gr = __shfl_sync(0xffffffffu, g_lane, j);
            const float dap = valid ? __uint_as_float(v[j]) : 0.0f;
            const float sg = 1.0f / (1.0f + __expf(-h));
            const float silu = h * sg;
            dgp[j] = dap * (silu * u);                     // <dA', a>, this lane's term
            const float da = gr * dap;
            const float dh = da * u * sg * (1.0f + h * (1.0f - sg));
            const float du = da * silu;
            if (valid) {
              const long long r = r0 + j;
              const __nv_bfloat16 hh = __float2bfloat16_rn(dh), uh = __float2bfloat16_rn(du);
              args.dhu_hi[r * twoI + i] = hh;
              args.dhu_lo[r * twoI + i] = __float2bfloat16_rn(dh - __bfloat162float(hh));
              args.dhu_hi[r * twoI + I + i] = uh;
              args.dhu_lo[r * twoI + I + i] = __float2bfloat16_rn(du - __bfloat162float(uh));
            }
            xb[j * C::XLD + lane] = dh;  // rows past the expert's end are zero (dap = 0)
            uv[j] = du;                  // u is no longer needed: keep du for the second pass
          }
          // dh | du along 2I for dX_g: each thread quantises its row's 32 indices (one MX block)
          const int p = p0 + lane;
          uint8_t* qrow = args.q + (long long)p * twoI;
          __syncwarp();
          mx_quantize_row32(xb + lane * C::XLD, qrow + (i - lane), args.qsf, S, p, s_h, kb_h);
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 32; ++j) xb[j * C::XLD + lane] = uv[j];
          __syncwarp();
          mx_quantize_row32(xb + lane * C::XLD, qrow + (I + i - lane), args.qsf, S, p, s_u, kb_u);
          __syncwarp();
          // partial gate gradient of each row over this CTA's 128 intermediate indices: lanes, then
          // warps in quarter order
          const float mine = warp_transpose_sum32(dgp, lane);  // row c*32 + lane, this warp's 32 indices
          dgbuf[quarter * 32 + lane] = mine;
          named_bar_sync(1, 128);
          if (quarter == 0 && lane < nr) {
            const float s4 = ((dgbuf[lane] + dgbuf[32 + lane]) + dgbuf[64 + lane]) + dgbuf[96 + lane];
            args.dg_part[((long long)t.row0 + c * 32 + lane) * nparts + part] = s4;
          }
          named_bar_sync(1, 128);  // dgbuf is free again
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty0_cl + 8u * acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or signals may still touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace mok
