// Weight-gradient GEMM of the expert FFN with a stationary operand (sm_103a, tcgen05).
//
//   out[e][n][m] = sum over the rows r of expert e of A[r][m] * B[r][n]
//
// with A [R][M] and B [R][N] row buffers (MN-major operands, K = the expert's rows).  One of
// the two operands is a bf16 hi + lo pair (the gradient dh|du or g*a, kept at ~16 significant
// bits); it is the larger load, so it stays in shared memory ("stationary") while the CTA walks a
// strip of 128 x 128 output tiles along the other dimension, and only the plain operand streams
// through the stage ring.  Each output tile therefore costs 16 KB of loads per 64 rows instead of
// 48 KB.  Experts with more rows than the stationary region holds (3 K blocks = 192 rows) are
// done tile by tile with the stationary K blocks reloaded in chunks.
//
// Strips are dealt dynamically: the producer warp takes the next strip index from a global
// counter and hands it to the MMA and epilogue warps through a 2-deep queue in shared memory.  On
// GB300 a static round-robin deal of this write-bound kernel ran at the pace of the slowest SMs
// (a store pattern like its epilogue's reached 6.7 TB/s dealt statically, 7.4-7.7 TB/s dealt from
// a counter).  Every strip is computed the same way whichever CTA takes it, so the results do not
// depend on the deal.
//
// Warps: 0 TMA producer, 1 MMA issuer, 2..9 epilogue in two groups of four, one per TMEM
// accumulator (TMEM -> registers 32 columns at a time, then coalesced stores: the output is
// transposed so that the 32 lanes of a warp, 32 consecutive m, write one 128-byte line per column).  The shared memory left by the stationary
// operand goes to a deep ring for the streaming operand: with only a few small K blocks per
// tile, the loads in flight, not the MMAs, bound the main loop (measured: 3 stages of 16 KB held
// the dW13 main loop at 4.6 ms on its own at the DSV3 layer).  All waits are bounded; the rows
// past an expert's end inside its last K block are zeroed in the stationary operand before the
// MMAs read it (the streaming operand's rows there then multiply zeros).
#pragma once
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace mok {

constexpr int WG_BK = 64;                    // rows per K block
constexpr int WG_KSTAT = 3;                  // K blocks the stationary region holds
constexpr int WG_STAT_SLOT = 4 * 8192;       // one K block of the stationary pair: hi (2 atoms), lo (2 atoms)
constexpr int WG_STAGE = 2 * 8192;           // one K block of the streaming operand (2 atoms)
constexpr int WG_STAGES = 7;
constexpr int WG_THREADS = 320;  // producer, MMA, two groups of four epilogue warps

struct WgradArgs {
  int M, N, E;              // output dims per expert (out[e][n][m]), experts
  const int* offsets;       // [E+1] expert row offsets
  void* out;                // [E][N][M] (fp32 or bf16)
  int* status;
  int* strip_counter;       // zero at launch: next strip to deal
};

__host__ __device__ constexpr size_t wgrad_smem_bytes(int E) {
  return size_t(WG_KSTAT) * WG_STAT_SLOT + size_t(WG_STAGES) * WG_STAGE + 1024 + 256 + size_t(E + 1) * 4;
}

// STAT_A: A is the stationary pair (tmA hi, tmA2 lo), strips walk n; otherwise B is (tmB, tmB2)
// and strips walk m.  OUT_F32: fp32 output, else bf16.  STAT_SPLIT false: the stationary
// operand is a single bf16 tensor (no lo half; the MXFP8 backward, whose operands are exact).
template <bool STAT_A, bool OUT_F32, bool STAT_SPLIT = true>
__global__ void __launch_bounds__(WG_THREADS, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                 const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                 const WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stat = smem;                                   // WG_KSTAT slots
  uint8_t* ring = stat + WG_KSTAT * WG_STAT_SLOT;         // WG_STAGES stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + WG_STAGES * WG_STAGE);
  // bars: full[S], empty[S], tfull[2], tempty[2], stat_full, stat_empty, drain, sq_full[2], sq_empty[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * WG_STAGES + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* sq = reinterpret_cast<volatile int*>(tmem_slot + 2);  // strip queue [2]
  int* s_off = reinterpret_cast<int*>(ring + WG_STAGES * WG_STAGE + 256);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[WG_STAGES + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * WG_STAGES + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * WG_STAGES + 2 + a]); };
  const uint32_t stat_full = smem_u32(&bars[2 * WG_STAGES + 4]);
  const uint32_t stat_empty = smem_u32(&bars[2 * WG_STAGES + 5]);
  const uint32_t drain_bar = smem_u32(&bars[2 * WG_STAGES + 6]);
  auto sq_full = [&](int d) { return smem_u32(&bars[2 * WG_STAGES + 7 + d]); };
  auto sq_empty = [&](int d) { return smem_u32(&bars[2 * WG_STAGES + 9 + d]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < WG_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(stat_full, 1);
    mbar_init(stat_empty, 1);
    mbar_init(drain_bar, 1);
    for (int d = 0; d < 2; ++d) {
      mbar_init(sq_full(d), 1);
      mbar_init(sq_empty(d), 9);  // the MMA warp and the 8 epilogue warps
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_off[i] = args.offsets[i];
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int MT = args.M / 128, NT = args.N / 128;
  const int per_e = STAT_A ? MT : NT;   // strips per expert
  const int strip_len = STAT_A ? NT : MT;
  const int total = args.E * per_e;
  // expert, fixed tile index, first row, rows, K blocks of strip s
  auto strip = [&](int s, int& e, int& f, int& row0, int& rows, int& nkb) {
    e = s / per_e;
    f = s - e * per_e;
    row0 = s_off[e];
    rows = s_off[e + 1] - row0;
    nkb = (rows + WG_BK - 1) / WG_BK;
  };
  // consumers (one warp): the next strip of the queue, -1 when none is left, -2 on abort
  int qd = 0;
  uint32_t qph = 0;
  auto take_strip = [&](int site) {
    int ok = 1, sv = -1;
    if (lane == 0) {
      ok = mbar_wait(sq_full(qd), qph, abort_flag, args.status, site, kWaitLimitNs, 64);
      if (ok) sv = *(sq + qd);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    sv = __shfl_sync(0xffffffffu, sv, 0);
    if (lane == 0 && ok) mbar_arrive(sq_empty(qd));
    __syncwarp();
    if (++qd == 2) {
      qd = 0;
      qph ^= 1;
    }
    return ok ? sv : -2;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmB2);
      const uint64_t pol = l2_policy_evict_last();
      const CUtensorMap* sh = STAT_A ? &tmA : &tmB;
      const CUtensorMap* sl = STAT_A ? &tmA2 : &tmB2;
      const CUtensorMap* st_map = STAT_A ? &tmB : &tmA;
      int stage = 0;
      uint32_t phase = 0, sphase = 0;
      bool ok = true;
      auto load_stat = [&](int f, int row0, int kb0, int nk) {
        if (!mbar_wait(stat_empty, sphase ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY, kWaitLimitNs, 32))
          return false;
        sphase ^= 1;
        mbar_arrive_expect_tx(stat_full, nk * (STAT_SPLIT ? WG_STAT_SLOT : WG_STAT_SLOT / 2));
        for (int j = 0; j < nk; ++j) {
          const uint32_t slot = smem_u32(stat + j * WG_STAT_SLOT);
          const int r = row0 + (kb0 + j) * WG_BK;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            tma_load_2d(slot + q * 8192, sh, stat_full, f * 128 + q * 64, r, pol);
            if (STAT_SPLIT) tma_load_2d(slot + 16384 + q * 8192, sl, stat_full, f * 128 + q * 64, r, pol);
          }
        }
        return true;
      };
      auto load_stream = [&](int i, int row0, int kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY, kWaitLimitNs, 32))
          return false;
        const uint32_t fb = full_bar(stage);
        const uint32_t sa = smem_u32(ring + stage * WG_STAGE);
        mbar_arrive_expect_tx(fb, WG_STAGE);
#pragma unroll
        for (int q = 0; q < 2; ++q) tma_load_2d(sa + q * 8192, st_map, fb, i * 128 + q * 64, row0 + kb * WG_BK, pol);
        if (++stage == WG_STAGES) {
          stage = 0;
          phase ^= 1;
        }
        return true;
      };
      while (ok) {
        // deal the next strip: take it from the counter and queue it for the other warps
        if (!mbar_wait(sq_empty(qd), qph ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY, kWaitLimitNs, 32))
          break;
        int s = atomicAdd(args.strip_counter, 1);
        if (s >= total) s = -1;
        *(sq + qd) = s;
        mbar_arrive(sq_full(qd));
        if (++qd == 2) {
          qd = 0;
          qph ^= 1;
        }
        if (s < 0) break;
        int e, f, row0, rows, nkb;
        strip(s, e, f, row0, rows, nkb);
        if (nkb == 0) continue;
        if (nkb <= WG_KSTAT) {
          ok = load_stat(f, row0, 0, nkb);
          for (int i = 0; i < strip_len && ok; ++i)
            for (int kb = 0; kb < nkb && ok; ++kb) ok = load_stream(i, row0, kb);
        } else {
          for (int i = 0; i < strip_len && ok; ++i)
            for (int kb0 = 0; kb0 < nkb && ok; kb0 += WG_KSTAT) {
              const int nk = min(WG_KSTAT, nkb - kb0);
              ok = load_stat(f, row0, kb0, nk);
              for (int kb = kb0; kb < kb0 + nk && ok; ++kb) ok = load_stream(i, row0, kb);
            }
        }
      }
      // on abort the loads in flight complete on their own barriers before the CTA's final sync
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, true, true);
    int stage = 0;
    uint32_t phase = 0, sphase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true, any = false;
    // waits for the stationary K blocks [kb0, kb0+nk) and zeroes the rows past the expert's end
    auto take_stat = [&](int rows, int kb0, int nk) {
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(stat_full, sphase, abort_flag, args.status, SITE_GEMM_MMA_FULL);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) return false;
      sphase ^= 1;
      tc_fence_after();
      const int last = kb0 + nk - 1;
      const int kvalid = rows - last * WG_BK;
      const int kend = (kvalid + 15) & ~15;
      if (kvalid < WG_BK && kvalid < kend) {
        uint8_t* slot = stat + (nk - 1) * WG_STAT_SLOT;
        const int nl = kend - kvalid;
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int idx = lane; idx < nl * 4 * 8; idx += 32) {
          const int chunk = idx & 7;
          const int li = idx >> 3;
          const int atom = li / nl;
          const int line = kvalid + (li - atom * nl);
          *reinterpret_cast<uint4*>(slot + atom * 8192 + line * 128 + chunk * 16) = z;
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      return true;
    };
    // MMAs of one K block: stationary slot j against the stage at the ring head
    auto mma_kblock = [&](int j, int rows, int kb, bool first) {
      int f_ok = 1;
      if (lane == 0) f_ok = mbar_wait(full_bar(stage), phase, abort_flag, args.status, SITE_GEMM_MMA_FULL);
      if (!__shfl_sync(0xffffffffu, f_ok, 0)) return false;
      tc_fence_after();
      if (lane == 0) {
        const int kvalid = min(WG_BK, rows - kb * WG_BK);
        const int nk16 = (kvalid + 15) >> 4;
        const uint32_t shi = smem_u32(stat + j * WG_STAT_SLOT);
        const uint32_t slo = shi + 16384;
        const uint32_t sst = smem_u32(ring + stage * WG_STAGE);
        const uint32_t d = tmem_base + acc * 128;
        for (int k16 = 0; k16 < nk16; ++k16) {
          const uint64_t dh = smem_desc_sw128(shi + k16 * 2048, MOK_MN_LBO, MOK_MN_SBO);
          const uint64_t dl = smem_desc_sw128(slo + k16 * 2048, MOK_MN_LBO, MOK_MN_SBO);
          const uint64_t ds = smem_desc_sw128(sst + k16 * 2048, MOK_MN_LBO, MOK_MN_SBO);
          const uint32_t accum = (first && k16 == 0) ? 0u : 1u;
          if (STAT_A) {
            umma_f16(d, dh, ds, idesc, accum);
            if (STAT_SPLIT) umma_f16(d, dl, ds, idesc, 1u);
          } else {
            umma_f16(d, ds, dh, idesc, accum);
            if (STAT_SPLIT) umma_f16(d, ds, dl, idesc, 1u);
          }
        }
        umma_commit(empty_bar(stage));
      }
      __syncwarp();
      any = true;
      if (++stage == WG_STAGES) {
        stage = 0;
        phase ^= 1;
      }
      return true;
    };
    auto begin_tile = [&]() {
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait(tempty_bar(acc), acc_phase ^ 1, abort_flag, args.status, SITE_GEMM_MMA_TMEM_EMPTY);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) return false;
      tc_fence_after();
      return true;
    };
    auto end_tile = [&]() {
      if (lane == 0) umma_commit(tfull_bar(acc));
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    };
    while (ok) {
      const int s = take_strip(SITE_GEMM_MMA_FULL);
      if (s < 0) break;
      int e, f, row0, rows, nkb;
      strip(s, e, f, row0, rows, nkb);
      if (nkb == 0) continue;
      if (nkb <= WG_KSTAT) {
        ok = take_stat(rows, 0, nkb);
        for (int i = 0; i < strip_len && ok; ++i) {
          ok = begin_tile();
          for (int kb = 0; kb < nkb && ok; ++kb) ok = mma_kblock(kb, rows, kb, kb == 0);
          if (ok) end_tile();
        }
        if (ok && lane == 0) umma_commit(stat_empty);  // the stationary slots are free once these MMAs end
        __syncwarp();
      } else {
        for (int i = 0; i < strip_len && ok; ++i) {
          ok = begin_tile();
          for (int kb0 = 0; kb0 < nkb && ok; kb0 += WG_KSTAT) {
            const int nk = min(WG_KSTAT, nkb - kb0);
            ok = take_stat(rows, kb0, nk);
            for (int kb = kb0; kb < kb0 + nk && ok; ++kb) ok = mma_kblock(kb - kb0, rows, kb, kb == 0);
            if (ok && lane == 0) umma_commit(stat_empty);
            __syncwarp();
          }
          if (ok) end_tile();
        }
      }
    }
    if (any) {
      if (lane == 0) {
        umma_commit(drain_bar);
        volatile int no_abort = 0;
        mbar_wait(drain_bar, 0, &no_abort, args.status, SITE_GEMM_DRAIN);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    // Two groups of four warps; group g drains accumulator g (the MMA alternates the two over
    // its tiles), keeping it until its stores are issued, so one group stores while the other
    // waits for the next tile: the store stream has no gap between tiles.
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    uint32_t acc_phase = 0;
    int tcount = 0;  // tiles with MMAs seen so far (both groups count all of them)
    bool ok = true;
    while (ok) {
      const int s = take_strip(SITE_GEMM_EPI_TMEM_FULL);
      if (s < 0) break;
      int e, f, row0, rows, nkb;
      strip(s, e, f, row0, rows, nkb);
      for (int i = 0; i < strip_len; ++i) {
        const int m = STAT_A ? f : i;
        const int n = STAT_A ? i : f;
        // out[e][n*128 + col][m*128 + quarter*32 + lane]
        const size_t base = (size_t)e * args.M * args.N + (size_t)(n * 128) * args.M + m * 128 + quarter * 32 + lane;
        if (nkb == 0) {
          // an expert without rows: its weight gradient is zero (the groups take alternate tiles)
          if ((i & 1) != grp) continue;
          for (int j = 0; j < 128; ++j) {
            if (OUT_F32) reinterpret_cast<float*>(args.out)[base + (size_t)j * args.M] = 0.0f;
            else reinterpret_cast<__nv_bfloat16*>(args.out)[base + (size_t)j * args.M] = __float2bfloat16_rn(0.0f);
          }
          continue;
        }
        const int acc = tcount & 1;
        ++tcount;
        if (acc != grp) continue;
        int w_ok = 1;
        if (lane == 0)
          w_ok = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, args.status, SITE_GEMM_EPI_TMEM_FULL, kWaitLimitNs,
                           256);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tacc = tmem_base + acc * 128 + (uint32_t(quarter * 32) << 16);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const size_t idx = base + (size_t)(c * 32 + j) * args.M;
            if (OUT_F32) reinterpret_cast<float*>(args.out)[idx] = __uint_as_float(v[j]);
            else reinterpret_cast<__nv_bfloat16*>(args.out)[idx] = __float2bfloat16_rn(__uint_as_float(v[j]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(acc));
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
}

}  // namespace mok
