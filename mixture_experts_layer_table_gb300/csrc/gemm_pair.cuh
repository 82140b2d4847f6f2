// CTA-pair grouped row GEMM for the expert FFN forward (sm_103a): GEMM1 x_g W13[e]^T with the
// SwiGLU epilogue, and GEMM2 a W2[e]^T (a as a bf16 hi / lo pair).
//
// Two CTAs of a cluster on neighbouring SMs run one 256 x 256 tile together with
// tcgen05.mma.cta_group::2: each CTA stages its own 128 rows of A and its half (128 columns)
// of B, the even CTA issues the MMAs, and each CTA's TMEM receives the accumulator of its own
// 128 rows.  Against the single-CTA 128 x 256 tile this halves the B bytes every SM loads and
// holds per MMA, which is what bounds the single-CTA kernel once the expert segments are long
// enough for the GEMM to be limited by the tensor cores rather than by the weight stream.
//
// Roles (both CTAs):   warp 0 TMA producer, warp 1 MMA issuer (even CTA only), warps 2..5
// epilogue (TMA tile stores from shared memory; see epi_*_tma).  Barriers:
//   full[s]   in the even CTA: one arrival (its producer, with the bytes of both CTAs) plus the
//             transaction bytes of both CTAs' loads (the loads name it across the pair)
//   empty[s]  in both CTAs: the MMA commit arrives on both when the stage has been read
//   tfull[a]  in both CTAs: the MMA commit arrives on both when accumulator a is complete
//   tempty[a] in the even CTA: 8 arrivals, the 4 epilogue warps of each CTA
// Tiles (expert e, column tile n, pair row tile m of 256 rows; m fastest) are dealt to the
// pairs round-robin in a fixed order, so results do not depend on timing; they are bitwise
// equal to the single-CTA kernel's (same K order, same fp32 accumulation per element).
#pragma once
#include "gemm.cuh"

namespace mok {

template <int EPI, int SPLIT>
struct PairCfg {
  static_assert(EPI == EPI_SWIGLU || EPI == EPI_F32, "pair GEMM epilogues");
  static_assert(SPLIT == SPLIT_NONE || SPLIT == SPLIT_A, "pair GEMM operands");
  static constexpr int BN = 256;                       // accumulator columns
  static constexpr int PM = 256;                       // rows of a pair tile
  static constexpr int A_TILES = SPLIT == SPLIT_A ? 2 : 1;
  static constexpr int B_HALF = 128 * BK * 2;          // this CTA's 128 B columns x 64 K
  static constexpr int STAGE_BYTES = A_TILE * A_TILES + B_HALF;
  static constexpr int PAIR_TX = 2 * STAGE_BYTES;      // bytes both CTAs' loads bring per stage
  // epilogue staging for TMA stores, per epilogue warp: SwiGLU h, u (4 KB each), a hi, lo
  // (2 KB each); fp32 output 4 KB
  static constexpr int STG_WARP = EPI == EPI_SWIGLU ? 12288 : 4096;
  static constexpr int STG_BYTES = 4 * STG_WARP;
  // 5 x 32 KB stages keep GEMM1's tensor cores as busy as 6 do (measured), which frees the room
  // for the staging buffers; GEMM2 keeps 4 x 48 KB
  static constexpr int STAGES = EPI == EPI_SWIGLU ? 5 : 4;
  static constexpr int TMEM_COLS = 2 * BN;
  static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                "tcgen05.alloc takes a power of two from 32 to 512 columns");
  static constexpr uint32_t IDESC = idesc_bf16_f32(PM, BN, false, false);
  static constexpr int THREADS = 192;
  static __host__ __device__ int n_tiles(const GemmArgs& a) {
    return EPI == EPI_SWIGLU ? a.I / 128 : (a.N + BN - 1) / BN;
  }
  static __host__ __device__ constexpr size_t smem_bytes(int E) {
    return size_t(STAGES) * STAGE_BYTES + STG_BYTES + 1024 /*align*/ + 256 /*barriers*/ + size_t(2) * (E + 1) * 4;
  }
};

struct PairTile {
  int e, n, m;
  int row0;  // first row of the 256-row pair tile
  int rows;  // valid rows of the pair tile (the tile may run past its expert)
  int mt;    // pair row tiles of this expert (they share each weight tile)
};

// Expert e owns pair tiles [ptoff[e]*NT, ptoff[e+1]*NT) with ptoff the prefix of ceil(rows/256).
__device__ __forceinline__ PairTile decode_pair_tile(int g, int NT, int E, const int* s_off, const int* s_ptoff) {
  int lo = 0, hi = E;  // largest e with s_ptoff[e]*NT <= g (the last of equal starts owns tiles)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_ptoff[mid] * NT <= g) lo = mid; else hi = mid;
  }
  PairTile t;
  t.e = lo;
  t.mt = s_ptoff[lo + 1] - s_ptoff[lo];
  const int local = g - s_ptoff[lo] * NT;
  t.n = local / t.mt;
  t.m = local - t.n * t.mt;
  t.row0 = s_off[lo] + t.m * 256;
  t.rows = min(256, s_off[lo + 1] - t.row0);
  return t;
}

template <int EPI, int SPLIT>
__global__ void __launch_bounds__(192, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                     const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmO0,
                     const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO2,
                     const GemmArgs args) {
  using C = PairCfg<EPI, SPLIT>;
  constexpr int STAGES = C::STAGES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + STAGES * STAGE_BYTES;  // C::STG_BYTES, 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::STG_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(staging + C::STG_BYTES + 256);
  int* s_ptoff = s_off + (args.E + 1);

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
  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_off[i] = args.offsets[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < args.E; ++e) {
      s_ptoff[e] = acc;
      acc += (s_off[e + 1] - s_off[e] + 255) >> 8;
    }
    s_ptoff[args.E] = acc;
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

  const int NT = C::n_tiles(args);
  const int total = s_ptoff[args.E] * NT;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if (SPLIT == SPLIT_A) tma_prefetch_desc(&tmA2);
      const uint64_t pol_act = l2_policy_evict_last();
      const uint64_t pol_once = l2_policy_evict_first();
      const uint64_t pol_shared = l2_policy_evict_normal();
      const uint32_t full0_cl = mapa_shared(full_bar(0), 0);  // the even CTA's full barriers
      const int nkb = args.K / BK;
      auto b_row_of = [&](const PairTile& t) {
        return (EPI == EPI_SWIGLU) ? (rank ? args.I : 0) + t.n * 128 : t.n * C::BN + 128 * (int)rank;
      };
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int g = pair; g < total && ok; g += npairs) {
        const PairTile t = decode_pair_tile(g, NT, args.E, s_off, s_ptoff);
        const uint64_t pol_w = t.mt > 1 ? pol_shared : pol_once;
        const int a_row = t.row0 + 128 * (int)rank;
        const int b_row = b_row_of(t);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait<true>(empty_bar(stage), phase ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY,
                               kWaitLimitNs, 32)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0_cl + 8u * stage;
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_TILE * C::A_TILES;
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), C::PAIR_TX);
          const int k0 = kb * BK;
          tma_load_2d_pair(sa, &tmA, fb, k0, a_row, pol_act);
          if (SPLIT == SPLIT_A) tma_load_2d_pair(sa + A_TILE, &tmA2, fb, k0, a_row, pol_act);
          tma_load_3d_pair(sb, &tmB, fb, k0, b_row, t.e, pol_w);
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
      const int nkb = args.K / BK;
      for (int g = pair; g < total && ok; g += npairs) {
        int w_ok = 1;
        if (lane == 0)
          w_ok = mbar_wait<true>(tempty_bar(acc), acc_phase ^ 1, abort_flag, args.status, SITE_GEMM_MMA_TMEM_EMPTY);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::BN;
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
            const uint32_t sb = sa + A_TILE * C::A_TILES;
#pragma unroll
            for (int k16 = 0; k16 < BK / 16; ++k16) {
              const uint64_t bdesc = smem_desc_sw128(sb + k16 * 32, 16, 1024);
              umma_f16_pair(d_tmem, smem_desc_sw128(sa + k16 * 32, 16, 1024), bdesc, C::IDESC,
                            (kb | k16) != 0 ? 1u : 0u);
              if (SPLIT == SPLIT_A)
                umma_f16_pair(d_tmem, smem_desc_sw128(sa + A_TILE + k16 * 32, 16, 1024), bdesc, C::IDESC, 1u);
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
    const int r_warp = 128 * (int)rank + quarter * 32;  // first row of this warp inside the pair tile
    uint8_t* stg = staging + (warp - 2) * C::STG_WARP;
    const uint32_t tempty0_cl = mapa_shared(tempty_bar(0), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int g = pair; g < total; g += npairs) {
      const PairTile t = decode_pair_tile(g, NT, args.E, s_off, s_ptoff);
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait<true>(tfull_bar(acc), acc_phase, abort_flag, args.status, SITE_GEMM_EPI_TMEM_FULL,
                               kWaitLimitNs, 256);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + acc * C::BN + (uint32_t(quarter * 32) << 16);
      const int nvalid = max(0, min(32, t.rows - r_warp));
      const long long row0 = (long long)(t.row0 + r_warp);
      if (EPI == EPI_SWIGLU) epi_swiglu_tma<true>(tacc, row0, nvalid, t.n, args, &tmO0, &tmO1, &tmO2, stg, lane);
      else epi_f32_tma<C::BN>(tacc, row0, nvalid, t.n, args, &tmO0, stg, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty0_cl + 8u * acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    // this warp's TMA stores have landed (and left shared memory) before the CTA exits
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
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
