// Weight-gradient GEMM on CTA pairs (sm_103a, tcgen05.mma.cta_group::2).
//
//   out[e][n][m] = sum over the rows r of expert e of A[r][m] * B[r][n]
//
// Same operands and roles as wgrad_kernel (wgrad.cuh): one operand (the bf16 hi + lo pair, or the
// plain one when neither is split) stays in shared memory for a strip of output tiles, the other
// streams through a 7-stage ring.  Here two CTAs on neighbouring SMs run 256 x 256 output tiles
// together: each CTA holds 128 columns of the stationary operand and streams 128 columns of the
// other, the even CTA issues M = 256, N = 256 MMAs that read both CTAs' halves, and each CTA's
// TMEM receives its 128 rows x 256 columns.  Per output element this halves the operand bytes
// each SM's tensor core reads from shared memory and the MMA instructions; at the DSV3 layer the
// single-CTA kernel's time followed its MMA count (half the MMAs: 10% faster) while the MMAs
// themselves run at the ideal rate in isolation.
//
// Warps (both CTAs): 0 TMA producer, 1 MMA issuer (even CTA) / stationary check (odd CTA), 2..9
// epilogue in two groups of four, one per TMEM accumulator.  The stationary region is a ring of
// WG_KSTAT slots of one 64-row K block each.  A block that ends inside an MMA K step (the last of
// an expert whose rows are not a multiple of 16) is loaded by each CTA onto its own full barrier;
// its warp 1 zeroes the rows past the expert's end and reports to the even CTA (ready, 2
// arrivals) before the pair's MMAs read the slot.  Every other block is loaded by both CTAs onto
// the even CTA's pfull barrier, as the streaming stages are, with no report (the report's round
// trip in every block held a long expert's pipeline: 16 experts of 1024 rows, dW13 2.02 ->
// 1.34 ms without it).  An expert of at most WG_KSTAT K blocks keeps its stationary
// blocks for the whole strip; a longer one streams them again for each tile, one block per slot,
// up to WG_KSTAT blocks ahead of the MMAs.
// Work items (tile pairs of the long experts, then strips of the others; see the item list
// below) go to whichever pair asks next; each output element is one tile's accumulator, reduced
// over the expert's rows in a fixed order, so results are bitwise those of the single-CTA kernel
// whichever pair computes them.
//
// The output leaves through TMA stores: an epilogue warp reads 32 columns of its 32 accumulator
// rows from TMEM, parks them in its 4 KB shared-memory block as 32 output rows of 32 elements
// and hands the block to a 2-D bulk tensor store (tmO: the output as [E*N rows][M], box 32 x 32),
// then goes on to the next 32 columns while the copy engine writes.  The warp releases its
// accumulator right after its last TMEM read, so that the next tile's MMAs need not wait for the
// stores.  (Plain stores from registers, 128 bytes a warp instruction, kept the accumulator until
// the last of them had issued: 5.5 TB/s of output at the DSV3 layer against 6.5 for the same
// store pattern alone.)  The operand ring is two stages shorter than the single-CTA kernel's to
// make room for the eight 4 KB blocks.
#pragma once
#include "wgrad.cuh"
#include "wgrad_items.h"

namespace mok {

constexpr int WGP_THREADS = 320;
// Streaming stages: six while the expert tables leave room (E <= WGP_E_SIX), else five.  A long
// expert's item needs two stages per K block (one per tile), so six keep three K blocks in
// flight, as many as the stationary ring holds.
constexpr int WGP_STAGES = 6;  // barriers are laid out for this many
constexpr int WGP_E_SIX = 284;
__host__ __device__ constexpr int wgp_stages(int E) { return E <= WGP_E_SIX ? 6 : 5; }
constexpr int WGP_STG = 4096;  // one epilogue warp's staging block (32 x 32 fp32)
// the barriers, the TMEM address, the abort flag and the item queue (WGP_TQ entries) share
// WGP_BAR_BYTES
constexpr int WGP_TQ = 4;
constexpr int WGP_BAR_BYTES = 336;
static_assert((2 * WGP_STAGES + 5 + 4 * WG_KSTAT + 2 * WGP_TQ) * 8 + 8 + WGP_TQ * 4 <= WGP_BAR_BYTES,
              "wgrad pair barriers");

// stationary slots, streaming stages, epilogue staging, alignment, barriers, the row offsets
// (i32 [E + 1]) and the expert list (u16 [E + 1])
__host__ __device__ constexpr size_t wgrad_pair_smem_bytes(int E) {
  return size_t(WG_KSTAT) * WG_STAT_SLOT + size_t(wgp_stages(E)) * WG_STAGE + 8 * size_t(WGP_STG) + 1024 + WGP_BAR_BYTES +
         size_t(E + 1) * 4 + size_t(E + 1) * 2;
}

template <bool STAT_A, bool OUT_F32, bool STAT_SPLIT = true>
__global__ void __launch_bounds__(WGP_THREADS, 1)
    wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                      const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                      const __grid_constant__ CUtensorMap tmO, const WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stat = smem;                                   // WG_KSTAT slots
  const int nst = wgp_stages(args.E);
  uint8_t* ring = stat + WG_KSTAT * WG_STAT_SLOT;         // nst stages
  uint8_t* stg_all = ring + nst * WG_STAGE;               // 8 epilogue warps x WGP_STG
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg_all + 8 * WGP_STG);
  // bars: full[S], empty[S], tfull[2], tempty[2], stat_full[K], stat_ready[K], stat_empty[K], drain,
  // stat_pfull[K] (K = WG_KSTAT), iq_full[Q], iq_empty[Q] (Q = WGP_TQ)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * WGP_STAGES + 5 + 4 * WG_KSTAT + 2 * WGP_TQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* iq = reinterpret_cast<volatile int*>(tmem_slot + 2);  // the item queue
  int* s_off = reinterpret_cast<int*>(stg_all + 8 * WGP_STG + WGP_BAR_BYTES);
  // experts with more than WG_KSTAT K blocks, then the others; [E] = how many are first
  uint16_t* s_list = reinterpret_cast<uint16_t*>(s_off + args.E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[WGP_STAGES + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * WGP_STAGES + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * WGP_STAGES + 2 + a]); };
  auto stat_full = [&](int j) { return smem_u32(&bars[2 * WGP_STAGES + 4 + j]); };
  auto stat_ready = [&](int j) { return smem_u32(&bars[2 * WGP_STAGES + 4 + WG_KSTAT + j]); };
  auto stat_empty = [&](int j) { return smem_u32(&bars[2 * WGP_STAGES + 4 + 2 * WG_KSTAT + j]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * WGP_STAGES + 4 + 3 * WG_KSTAT]);
  // a stationary block loaded by both CTAs onto the even CTA's barrier (no rows to zero)
  auto stat_pfull = [&](int j) { return smem_u32(&bars[2 * WGP_STAGES + 5 + 3 * WG_KSTAT + j]); };
  // the item queue: full in both CTAs, empty in the even CTA
  auto iq_full = [&](int q) { return smem_u32(&bars[2 * WGP_STAGES + 5 + 4 * WG_KSTAT + q]); };
  auto iq_empty = [&](int q) { return smem_u32(&bars[2 * WGP_STAGES + 5 + 4 * WG_KSTAT + WGP_TQ + q]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);  // the 4 warps of group a in both CTAs
    }
    for (int j = 0; j < WG_KSTAT; ++j) {
      mbar_init(stat_full(j), 1);
      mbar_init(stat_ready(j), 2);  // warp 1 of both CTAs
      mbar_init(stat_empty(j), 1);
      mbar_init(stat_pfull(j), 1);
    }
    for (int q = 0; q < WGP_TQ; ++q) {
      mbar_init(iq_full(q), 1);
      // readers: the even CTA's MMA warp and epilogue warps, the odd CTA's producer, warp 1 and
      // epilogue warps
      mbar_init(iq_empty(q), 1 + 8 + 1 + 1 + 8);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_off[i] = args.offsets[i];
  if (warp == 2) {
    // the expert list: first the experts whose rows exceed the stationary region (in expert
    // order), then the others (in expert order); s_list[E] = how many are first
    int n_long = 0;
    for (int pass = 0; pass < 2; ++pass) {
      int at = pass == 0 ? 0 : n_long;
      for (int e0 = 0; e0 < args.E; e0 += 32) {
        const int e = e0 + lane;
        const bool is_long = e < args.E && args.offsets[e + 1] - args.offsets[e] > WG_KSTAT * WG_BK;
        const bool take = e < args.E && (pass == 0 ? is_long : !is_long);
        const uint32_t m = __ballot_sync(0xffffffffu, take);
        if (take) s_list[at + __popc(m & ((1u << lane) - 1u))] = (uint16_t)e;
        at += __popc(m);
      }
      if (pass == 0) n_long = at;
    }
    if (lane == 0) s_list[args.E] = (uint16_t)n_long;
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // 256-wide tiles of the pair; this CTA owns the 128 columns at +128*rank of each
  const int MT = args.M / 256, NT = args.N / 256;
  const int per_e = STAT_A ? MT : NT;   // strips per expert
  const int strip_len = STAT_A ? NT : MT;
  // Work items, in two lists:
  //  * one item per two neighbouring output tiles (i, i + 1) of one stationary strip f of
  //    each expert with more than WG_KSTAT K blocks of rows (expert by expert, in s_list order).
  //    Their stationary blocks are streamed again for every item, so the pairs spread over the
  //    items of one expert at a time and share its rows in L2 (one pair per strip of 28 tiles, as
  //    the strips below are dealt, kept some five long experts in flight at once, more than L2
  //    holds: at 16 experts of 1024 rows, 45% of the operand reads hit L2 and dW13 took 2.3 us
  //    per 64-row K block of a pair tile; tile by tile over one expert, 1.6 us).  Both tiles
  //    accumulate at once, one in each TMEM accumulator, so each stationary block that arrives
  //    feeds twice the MMAs (the epilogue of an item then no longer overlaps its MMAs; at 16
  //    experts of 1024 rows dW13 2.59 -> 2.02 ms, 1.34 us per K block of a pair tile);
  //  * one item per strip (expert, 256-wide stationary tile f, all strip_len tiles) of the
  //    other experts, whose stationary blocks stay in shared memory for the whole strip (each
  //    expert's strips in a row, so neighbouring pairs share its streaming rows in L2).
  // The two lists are merged with the long experts' items spread evenly among the strips, each
  // list in its own order: the long experts' items are bound by their MMAs, the strips by their
  // output stores, so pairs running both kinds at once keep the tensor cores and HBM busy together
  // (the long items all first: skewed DSV3 layer dW13 5.99 ms, merged 5.74).  The pairs take
  // positions of the merged list in order from one counter (args.strip_counter): a pair that
  // draws costly items, or runs on slower SMs, simply takes fewer (a fixed back-and-forth deal
  // held the whole launch to the slowest pair's share).  The even CTA's producer takes each item
  // and passes its index to every role of both CTAs through a WGP_TQ-deep queue in shared memory;
  // -1 ends it.  Which pair computes an output tile does not change it.
  const WgpItems wi = wgp_items(per_e, strip_len, s_list[args.E], args.E);
  const int total = wi.total;
  // item -> expert e, stationary strip f, tiles [i0, i1) along the strip, its rows
  auto item = [&](int n, int& e, int& f, int& i0, int& i1, int& row0, int& rows, int& nkb) {
    int le;
    wgp_item(wi, n, le, f, i0, i1);
    e = s_list[le];
    row0 = s_off[e];
    rows = s_off[e + 1] - row0;
    nkb = (rows + WG_BK - 1) / WG_BK;
  };
  const int half0 = 128 * (int)rank;
  // K block kb of an expert with `rows` rows ends inside an MMA K step: the stationary rows past
  // the expert's end must be zeroed before the MMAs read them (each CTA its own, then a report)
  auto stat_ragged = [&](int rows, int kb) {
    const int kvalid = rows - kb * WG_BK;
    return kvalid < WG_BK && (kvalid & 15) != 0;
  };
  // the q-th item of this pair (-1: no more): taken by the even CTA's producer (one thread) ...
  auto publish_item = [&](int q, int& n) -> bool {
    const int qs = q % WGP_TQ;
    const uint32_t u = (uint32_t)(q / WGP_TQ) & 1u;
    if (!mbar_wait<true>(iq_empty(qs), u ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY, kWaitLimitNs, 32))
      return false;
    const int pos = atomicAdd(args.strip_counter, 1);
    n = pos < total ? wgp_item_at(wi, pos) : -1;  // the long experts' items spread among the strips
    iq[qs] = n;
    st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(&iq[qs])), 1), (uint32_t)n);
    mbar_arrive(iq_full(qs));
    mbar_arrive_cluster(mapa_shared(iq_full(qs), 1));  // release: the peer's copy is written
    return true;
  };
  // ... and read by every other role (lane 0 of a warp, or one thread), which counts itself out
  auto read_item = [&](int q, int& n, uint32_t sleep_ns, bool warp_wide) -> bool {
    const int qs = q % WGP_TQ;
    const uint32_t u = (uint32_t)(q / WGP_TQ) & 1u;
    int w_ok = 1;
    if (lane == 0 || !warp_wide) {
      w_ok = mbar_wait<true>(iq_full(qs), u, abort_flag, args.status, SITE_GEMM_MMA_FULL, kWaitLimitNs, sleep_ns);
      if (w_ok) {
        n = iq[qs];
        if (rank == 0) mbar_arrive(iq_empty(qs));
        else mbar_arrive_cluster(mapa_shared(iq_empty(qs), 0));
      }
    }
    if (warp_wide) {
      w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      n = __shfl_sync(0xffffffffu, n, 0);
    }
    return w_ok != 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmB2);
      const uint64_t pol = l2_policy_evict_last();
      const CUtensorMap* sh = STAT_A ? &tmA : &tmB;
      const CUtensorMap* sl = STAT_A ? &tmA2 : &tmB2;
      const CUtensorMap* st_map = STAT_A ? &tmB : &tmA;
      const uint32_t full0_cl = mapa_shared(full_bar(0), 0);  // the even CTA's full barriers
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      int sc = 0;  // stationary K blocks loaded so far: the next goes to slot sc % WG_KSTAT
      uint32_t hs_ph = 0, pf_ph = 0;  // per slot: phase bits of its full and its pfull barrier
      uint32_t last_pair = 0, last_ph = 0;  // per slot: its latest load's barrier kind and phase
      const uint32_t pfull0_cl = mapa_shared(stat_pfull(0), 0);
      bool ok = true;
      auto load_stat = [&](int f, int row0, int rows, int kb) {
        const int j = sc % WG_KSTAT;
        const uint32_t ph = (uint32_t)(sc / WG_KSTAT) & 1u;
        if (!mbar_wait<true>(stat_empty(j), ph ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY,
                             kWaitLimitNs, 32))
          return false;
        const uint32_t bytes = STAT_SPLIT ? WG_STAT_SLOT : WG_STAT_SLOT / 2;
        const uint32_t slot = smem_u32(stat + j * WG_STAT_SLOT);
        const int r = row0 + kb * WG_BK;
        const uint32_t bit = 1u << j;
        if (stat_ragged(rows, kb)) {
          // rows past the expert's end to zero: each CTA's bytes on its own barrier
          mbar_arrive_expect_tx(stat_full(j), bytes);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            tma_load_2d(slot + q * 8192, sh, stat_full(j), f * 256 + half0 + q * 64, r, pol);
            if (STAT_SPLIT) tma_load_2d(slot + 16384 + q * 8192, sl, stat_full(j), f * 256 + half0 + q * 64, r, pol);
          }
          last_pair &= ~bit;
          last_ph = (last_ph & ~bit) | (hs_ph & bit);
          hs_ph ^= bit;
        } else {
          // both CTAs' bytes on the even CTA's barrier, as the streaming stages
          if (rank == 0) mbar_arrive_expect_tx(stat_pfull(j), 2 * bytes);
          const uint32_t pb = pfull0_cl + 8u * j;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            tma_load_2d_pair(slot + q * 8192, sh, pb, f * 256 + half0 + q * 64, r, pol);
            if (STAT_SPLIT) tma_load_2d_pair(slot + 16384 + q * 8192, sl, pb, f * 256 + half0 + q * 64, r, pol);
          }
          last_pair |= bit;
          last_ph = (last_ph & ~bit) | (pf_ph & bit);
          pf_ph ^= bit;
        }
        ++sc;
        return true;
      };
      auto load_stream = [&](int i, int row0, int kb) {
        if (!mbar_wait<true>(empty_bar(stage), phase ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY,
                             kWaitLimitNs, 32))
          return false;
        const uint32_t fb = full0_cl + 8u * stage;
        const uint32_t sa = smem_u32(ring + stage * WG_STAGE);
        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * WG_STAGE);
#pragma unroll
        for (int q = 0; q < 2; ++q)
          tma_load_2d_pair(sa + q * 8192, st_map, fb, i * 256 + half0 + q * 64, row0 + kb * WG_BK, pol);
        ++issued;
        if (++stage == nst) {
          stage = 0;
          phase ^= 1;
        }
        return true;
      };
      for (int q = 0; ok; ++q) {
        int n = -1;
        ok = rank == 0 ? publish_item(q, n) : read_item(q, n, 32, false);
        if (!ok || n < 0) break;
        int e, f, i0, i1, row0, rows, nkb;
        item(n, e, f, i0, i1, row0, rows, nkb);
        if (nkb == 0) continue;
        if (nkb <= WG_KSTAT) {
          for (int kb = 0; kb < nkb && ok; ++kb) ok = load_stat(f, row0, rows, kb);
          for (int i = i0; i < i1 && ok; ++i)
            for (int kb = 0; kb < nkb && ok; ++kb) ok = load_stream(i, row0, kb);
        } else {
          for (int kb = 0; kb < nkb && ok; ++kb) {
            ok = load_stat(f, row0, rows, kb);
            for (int i = i0; i < i1 && ok; ++i) ok = load_stream(i, row0, kb);
          }
        }
      }
      if (!ok) {
        // Aborted: let no copy land in shared memory after the CTA has left.  The even CTA's full
        // barriers count both CTAs' stream bytes; the peer cannot observe its own and waits a while.
        volatile int no_abort = 0;
        // the latest stationary load of each slot: on this CTA's own barrier, or (pair form) on the
        // even CTA's, which counts both CTAs' bytes; the odd CTA waits a while below
        for (int j = 0; j < min(sc, WG_KSTAT); ++j) {
          const uint32_t bit = 1u << j;
          const uint32_t lp = (last_ph >> j) & 1u;
          if (!(last_pair & bit)) mbar_wait(stat_full(j), lp, &no_abort, args.status, SITE_GEMM_DRAIN);
          else if (rank == 0) mbar_wait(stat_pfull(j), lp, &no_abort, args.status, SITE_GEMM_DRAIN);
        }
        if (rank == 0) {
          const int outstanding = min(issued, nst);
          int st = stage;
          uint32_t ph = phase;
          for (int n = 0; n < outstanding; ++n) {
            if (--st < 0) {
              st = nst - 1;
              ph ^= 1;
            }
            mbar_wait(full_bar(st), ph, &no_abort, args.status, SITE_GEMM_DRAIN);
          }
        } else {
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 100000ull) __nanosleep(1000);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_bf16_f32(256, 256, true, true);
    int stage = 0;
    uint32_t phase = 0;
    int sc = 0;  // stationary K blocks taken so far, in the producer's order
    uint32_t hs_ph = 0, pf_ph = 0;  // per slot: phase bits of its full / ready and its pfull barrier
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true, any = false;
    // Stationary K block kb of the item, in slot sc % WG_KSTAT (returned in j).  Pair form: the even
    // CTA waits for both CTAs' bytes on its pfull barrier.  Ragged form: each CTA waits for its own
    // bytes, zeroes its rows past the expert's end and reports to the even CTA, which waits for both
    // reports.
    auto take_stat = [&](int rows, int kb, int& j) {
      j = sc % WG_KSTAT;
      ++sc;
      const uint32_t bit = 1u << j;
      int w_ok = 1;
      if (!stat_ragged(rows, kb)) {
        const uint32_t ph = (pf_ph >> j) & 1u;
        pf_ph ^= bit;
        if (rank == 0) {
          if (lane == 0) w_ok = mbar_wait<true>(stat_pfull(j), ph, abort_flag, args.status, SITE_GEMM_MMA_FULL);
          if (!__shfl_sync(0xffffffffu, w_ok, 0)) return false;
          tc_fence_after();
        }
        return true;
      }
      const uint32_t ph = (hs_ph >> j) & 1u;
      hs_ph ^= bit;
      if (lane == 0) w_ok = mbar_wait(stat_full(j), ph, abort_flag, args.status, SITE_GEMM_MMA_FULL);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) return false;
      {
        const int kvalid = rows - kb * WG_BK;
        const int kend = (kvalid + 15) & ~15;
        uint8_t* slot = stat + j * WG_STAT_SLOT;
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
      if (lane == 0) mbar_arrive_cluster(mapa_shared(stat_ready(j), 0));
      if (rank == 0) {
        if (lane == 0)
          w_ok = mbar_wait<true>(stat_ready(j), ph, abort_flag, args.status, SITE_GEMM_MMA_FULL);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) return false;
        tc_fence_after();
      }
      return true;
    };
    auto mma_kblock = [&](int j, int rows, int kb, bool first, int next = 0) {
      int f_ok = 1;
      if (lane == 0) f_ok = mbar_wait<true>(full_bar(stage), phase, abort_flag, args.status, SITE_GEMM_MMA_FULL);
      if (!__shfl_sync(0xffffffffu, f_ok, 0)) return false;
      tc_fence_after();
      if (lane == 0) {
        const int kvalid = min(WG_BK, rows - kb * WG_BK);
        const int nk16 = (kvalid + 15) >> 4;
        const uint32_t shi = smem_u32(stat + j * WG_STAT_SLOT);
        const uint32_t slo = shi + 16384;
        const uint32_t sst = smem_u32(ring + stage * WG_STAGE);
        const uint32_t d = tmem_base + (acc ^ next) * 256;
        for (int k16 = 0; k16 < nk16; ++k16) {
          const uint64_t dh = smem_desc_sw128(shi + k16 * 2048, MOK_MN_LBO, MOK_MN_SBO);
          const uint64_t dl = smem_desc_sw128(slo + k16 * 2048, MOK_MN_LBO, MOK_MN_SBO);
          const uint64_t ds = smem_desc_sw128(sst + k16 * 2048, MOK_MN_LBO, MOK_MN_SBO);
          const uint32_t accum = (first && k16 == 0) ? 0u : 1u;
          if (STAT_A) {
            umma_f16_pair(d, dh, ds, idesc, accum);
            if (STAT_SPLIT) umma_f16_pair(d, dl, ds, idesc, 1u);
          } else {
            umma_f16_pair(d, ds, dh, idesc, accum);
            if (STAT_SPLIT) umma_f16_pair(d, ds, dl, idesc, 1u);
          }
        }
        umma_commit_pair(empty_bar(stage), 0x3);
      }
      __syncwarp();
      any = true;
      if (++stage == nst) {
        stage = 0;
        phase ^= 1;
      }
      return true;
    };
    // next = 1: the tile after the current one (the other accumulator; its use count is one more
    // when the current one is accumulator 1)
    auto begin_tile = [&](int next = 0) {
      const int a = acc ^ next;
      const uint32_t ph = (next && acc == 1) ? acc_phase ^ 1 : acc_phase;
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait<true>(tempty_bar(a), ph ^ 1, abort_flag, args.status, SITE_GEMM_MMA_TMEM_EMPTY);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) return false;
      tc_fence_after();
      return true;
    };
    auto end_tile = [&]() {
      if (lane == 0) umma_commit_pair(tfull_bar(acc), 0x3);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    };
    auto release_stat = [&](int j) {
      if (lane == 0) umma_commit_pair(stat_empty(j), 0x3);  // both CTAs' slots are free once these MMAs end
      __syncwarp();
    };
    for (int q = 0; ok; ++q) {
      int n = -1;
      ok = read_item(q, n, 32, true);
      if (!ok || n < 0) break;
      int e, f, i0, i1, row0, rows, nkb;
      item(n, e, f, i0, i1, row0, rows, nkb);
      if (nkb == 0) continue;
      if (nkb <= WG_KSTAT) {
        int js[WG_KSTAT];
        for (int kb = 0; kb < nkb && ok; ++kb) ok = take_stat(rows, kb, js[kb]);
        if (rank == 0) {
          for (int i = i0; i < i1 && ok; ++i) {
            ok = begin_tile();
            for (int kb = 0; kb < nkb && ok; ++kb) ok = mma_kblock(js[kb], rows, kb, kb == 0);
            if (ok) end_tile();
          }
          for (int kb = 0; kb < nkb && ok; ++kb) release_stat(js[kb]);
        }
      } else {
        // tiles i0 and i0 + 1 (if any) in the accumulators acc and acc ^ 1, K block by K block
        const int nt = i1 - i0;
        if (rank == 0) {
          ok = begin_tile();
          if (ok && nt == 2) ok = begin_tile(1);
        }
        for (int kb = 0; kb < nkb && ok; ++kb) {
          int j;
          ok = take_stat(rows, kb, j);
          if (ok && rank == 0) {
            ok = mma_kblock(j, rows, kb, kb == 0);
            if (ok && nt == 2) ok = mma_kblock(j, rows, kb, kb == 0, 1);
            if (ok) release_stat(j);
          }
        }
        if (ok && rank == 0) {
          end_tile();
          if (nt == 2) end_tile();
        }
      }
    }
    if (rank == 0 && any) {
      if (lane == 0) {
        umma_commit_pair(drain_bar, 0x1);
        volatile int no_abort = 0;
        mbar_wait(drain_bar, 0, &no_abort, args.status, SITE_GEMM_DRAIN);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    // Two groups of four warps; group g drains accumulator g of this CTA (its 128 rows x 256
    // columns) and then reports to the even CTA.
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const uint32_t tempty0_cl = mapa_shared(tempty_bar(0), 0);
    uint8_t* stg = stg_all + (warp - 2) * WGP_STG;
    const uint32_t stg_u = smem_u32(stg);
    if (lane == 0) tma_prefetch_desc(&tmO);
    // the output is written once and not read back here: its lines go first when L2 needs room,
    // before the operand rows that the other strips of the expert read again
    const uint64_t pol_out = l2_policy_evict_first();
    uint32_t acc_phase = 0;
    int tcount = 0;  // tiles with MMAs seen so far (both groups count all of them)
    bool ok = true;
    for (int q = 0; ok; ++q) {
      int n = -1;
      if (!read_item(q, n, 256, true) || n < 0) break;
      int e, f, i0, i1, row0, rows, nkb;
      item(n, e, f, i0, i1, row0, rows, nkb);
      for (int i = i0; i < i1; ++i) {
        // this CTA's rows m and the tile's columns n (256)
        const int m0 = (STAT_A ? f : i) * 256 + half0;
        const int n0 = (STAT_A ? i : f) * 256;
        // out[e][n0 + col][m0 + quarter*32 + lane]
        const size_t base = (size_t)e * args.M * args.N + (size_t)n0 * args.M + m0 + quarter * 32 + lane;
        if (nkb == 0) {
          // an expert without rows: its weight gradient is zero (the groups take alternate tiles)
          if ((i & 1) != grp) continue;
          for (int j = 0; j < 256; ++j) {
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
          w_ok = mbar_wait<true>(tfull_bar(acc), acc_phase, abort_flag, args.status, SITE_GEMM_EPI_TMEM_FULL,
                                 kWaitLimitNs, 256);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tacc = tmem_base + acc * 256 + (uint32_t(quarter * 32) << 16);
        const int out_m = m0 + quarter * 32;           // the store box's first column (m)
        const int out_r = e * args.N + n0;             // the tile's first row (n) of the [E*N][M] view
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + c * 32, v);
          tmem_wait_ld();
          if (c == 7) {
            // the accumulator has been read: the next tile's MMAs may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(tempty0_cl + 8u * acc);
          }
          if (lane == 0) bulk_wait_group_read<0>();  // the previous block's store has read the buffer
          __syncwarp();
          // row j of the block = output row n0 + 32c + j, column lane = m (128 or 64 bytes a row)
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (OUT_F32) reinterpret_cast<float*>(stg)[j * 32 + lane] = __uint_as_float(v[j]);
            else reinterpret_cast<__nv_bfloat16*>(stg)[j * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[j]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d_hint(&tmO, stg_u, out_m, out_r + c * 32, pol_out);
            bulk_commit_group();
          }
        }
        acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait_group_all();  // every block has been written (and its buffer read)
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or signals may still touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

}  // namespace mok
