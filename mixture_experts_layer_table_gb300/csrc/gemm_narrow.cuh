// Narrow-segment grouped GEMM on CTA pairs (sm_103a): out[r][j] = sum_k X[r][k] W[e][j][k] over
// the expert-sorted rows r of each expert e, computed transposed: D[j][r] = W[e] X^T.
//
// The row-tile kernels (gemm.cuh, gemm_pair.cuh) put an expert's rows on the MMA's M side in
// tiles of 128 (or 256) rows; with about 128 rows per expert, half the experts spill a few rows
// into a second tile and the tensor cores spend a third of their work on padding, twice over
// for a hi / lo operand.  Here the roles swap: 256 weight rows (output columns j) are the M of a
// tcgen05.mma.cta_group::2 (128 per CTA of the pair) and the expert's rows are its N, a multiple
// of 16 up to 256, so an expert pads to 16 rows.  An expert with more than 256 rows is cut into
// equal chunks (multiples of 16).  Per SM and 64-deep K step the pair loads 16 KB of weights and
// at most 16 KB of rows per operand, against 32 KB of weights + 16 KB per A operand for the
// single-CTA row tile.  Results are bitwise equal to the row-tile kernels' (same K order, same
// fp32 accumulation per element).
//
//   WMN = false  W K-major  [E][N][K]   (GEMM2: o = a W2[e]^T, K = I)
//   WMN = true   W MN-major [E][K][N]   (dX_g = dHU W13[e], K = 2I)
//   SPLIT        X is a bf16 hi / lo pair, two MMAs per K step into the same accumulator
//   EPI_SWIGLU   GEMM1 x_g W13[e]^T (K = H): each CTA's 128 weight rows are 64 gate rows and the
//                64 up rows of the same intermediate indices, so h and u of one (row, i) sit on
//                TMEM lane quarters q and q + 2; the gate warp hands h to the up warp through
//                shared memory, which forms a = silu(h) u (stored as a bf16 hi / lo pair, or with
//                args.a_f16 as one fp16 value, for a GEMM2 on fp16 operands).
//   args.f16     the MMA operands are fp16 (GEMM2 on an fp16 copy of W2 and fp16 a) instead of bf16.
//
// Roles (both CTAs): warp 0 TMA producer, warp 1 MMA issuer (even CTA only), warps 2..5 epilogue
// (tcgen05.ld of 32 rows x 32 columns, then per row one 128-byte store of 32 consecutive
// columns by the warp).  Barriers as in gemm_pair.cuh: full[s] in the even CTA (one arrival with
// the bytes of both CTAs), empty[s] and tfull[a] in both CTAs (multicast commits), tempty[a] in
// the even CTA (8 arrivals).  Tiles (expert e, weight tile m of 256 columns, row chunk c; c
// fastest, then m, so the pairs running one expert at the same time share its rows and each
// weight tile in L2) are taken by the pairs in that order from one counter (or, without a
// counter, dealt round-robin); every output element is one tile's accumulator, reduced over K in
// a fixed order, whichever pair computes it.
#pragma once
#include <type_traits>

#include "combine.cuh"
#include "gemm.cuh"
#include "narrow_tiles.h"

namespace mok {

// Shared memory after the stages and the SwiGLU exchange buffer: barriers, TMEM address, abort
// flag and the tile queue: NARROW_TQ entries of NARROW_QE ints at byte NARROW_QOFF (the deep
// form below packs them tighter).
constexpr int NARROW_BAR_BYTES = 1024;
constexpr int NARROW_TQ = 8;
constexpr int NARROW_QE = 12;
constexpr int NARROW_QOFF = 512;
// Experts the deep form's 16-bit chunk prefixes and smem budget allow.
constexpr int NARROW_DEEP_MAX_E = 256;

template <bool WMN, bool SPLIT, int NMAX_, int EPI = EPI_F32>
struct NarrowCfg {
  static_assert(EPI == EPI_F32 || EPI == EPI_F32_PAIRED ||
                    ((EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_PAIRED) && !WMN && !SPLIT),
                "narrow GEMM epilogues");
  // EPI_SWIGLU_PAIRED: each CTA's A is 128 gate rows and the 128 up rows of the same intermediate
  // indices, two MMAs per K step (gate, up) share the row operand, h and u accumulate in columns
  // [0, N) and [256, 256 + N) of one accumulator (no second one: the epilogue is not overlapped).
  // EPI_F32_PAIRED: each CTA's A is its 128 rows of two weight tiles 256 rows apart (a pair tile
  // covers 512 output columns), the same two-MMA arrangement.
  static constexpr bool kPaired = EPI == EPI_SWIGLU_PAIRED || EPI == EPI_F32_PAIRED;
  static constexpr int ACCS = kPaired ? 1 : 2;  // accumulators in TMEM
  static constexpr int PM = 256;                // weight rows (output columns) of a pair tile
  static constexpr int NMAX = NMAX_;            // rows of a pair tile at most
  // narrow_x_boxes(h) <= NMAX / 2 for every h <= NMAX / 2 when NMAX / 2 is a multiple of 32
  static_assert((NMAX / 2) % NARROW_XBOX_S == 0, "the boxes of one CTA's rows fit its X buffer");
  static constexpr int X_OP = (NMAX / 2) * 128; // one CTA's rows of one X operand x 64 K
  static constexpr int A_BYTES = (kPaired ? 2 : 1) * 128 * BK * 2;
  static constexpr int X_OPS = SPLIT ? 2 : 1;
  static constexpr int STAGE_BYTES = A_BYTES + X_OPS * X_OP;
  // The deep form: the paired split-operand GEMMs (GEMM2, dX_g) in 192-row chunks take a fourth
  // 56 KB stage (measured at the DSV3 layer, 128 rows per expert: GEMM2 1.556 -> 1.473 ms, dX_g
  // 2.749 -> 2.717 ms), which fits beside the alignment pad only with a 4-entry tile queue packed
  // after the barriers and 16-bit chunk prefixes, for at most NARROW_DEEP_MAX_E experts.
  static constexpr bool kDeep = EPI == EPI_F32_PAIRED && SPLIT && NMAX == 192;
  static constexpr int STAGES = kDeep ? 4 : (208 * 1024 / STAGE_BYTES) < 8 ? (208 * 1024 / STAGE_BYTES) : 8;
  static constexpr int TQ = kDeep ? 4 : NARROW_TQ;
  static constexpr int QOFF = kDeep ? 192 : NARROW_QOFF;
  static constexpr int BAR_BYTES = kDeep ? 384 : NARROW_BAR_BYTES;
  using coff_t = typename std::conditional<kDeep, uint16_t, int>::type;
  // two accumulators of NMAX columns (paired: one of 256 + NMAX); tcgen05.alloc takes a power of
  // two from 32 to 512
  static constexpr int TMEM_COLS = (kPaired || 2 * NMAX > 256) ? 512 : 256;
  static_assert(NMAX % 32 == 0 && NMAX >= 32 && 2 * NMAX <= 512, "accumulators must fit the TMEM allocation");
  // epilogue warps: two per TMEM lane quarter in the paired SwiGLU form (taking alternate 8-row
  // blocks), whose single accumulator is held while the epilogue stores h, u and a: more warps
  // storing at once free it sooner (at T = 16384, 512 rows per expert, the stores of four warps
  // held the MMAs 0.8 ms of 6.0)
  static constexpr int EPI_WARPS = EPI == EPI_SWIGLU_PAIRED ? 8 : 4;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  // SwiGLU: one 32 x 32 fp32 block of h and one of u per pair of warps
  static constexpr int XBUF_BYTES = EPI == EPI_SWIGLU ? 2 * 2 * 32 * 32 * 4 : 0;
  // weight tiles: 256 output columns, or (SwiGLU) 128 intermediate indices (gate and up rows),
  // or (paired) 256 intermediate indices
  static __host__ __device__ int m_tiles(const GemmArgs& a) {
    return EPI == EPI_SWIGLU_PAIRED ? a.I / 256
           : EPI == EPI_SWIGLU     ? a.I / 128
           : EPI == EPI_F32_PAIRED ? (a.N + 2 * PM - 1) / (2 * PM)
                                   : (a.N + PM - 1) / PM;
  }
  // stages, exchange buffer, alignment pad, barriers, row offsets (i32 [E + 1]), chunk prefixes
  static __host__ __device__ constexpr size_t smem_bytes(int E) {
    return size_t(STAGES) * STAGE_BYTES + XBUF_BYTES + 1024 /*align*/ + BAR_BYTES + size_t(E + 1) * 4 +
           ((size_t(E + 1) * sizeof(coff_t) + 3) & ~size_t(3));
  }
};

// tmX / tmX2: X hi / lo in 64-row boxes; tmXs / tmX2s: the same in 32-row boxes.  tmW (SwiGLU):
// W13 seen as [E][2][I][H], one box = 64 gate rows and their 64 up rows.
//
// RING (GEMM1 of the ring forward): X is the token ring [slots * mb_rows][H].  Every CTA first
// copies minibatch 0 into the ring (ring_gather_first); then the first args.comm_ctas CTAs (an
// even number, whole clusters) gather the later minibatches (ring_gather, as in gemm.cuh) while
// the CTA pairs run the narrow tiles of each minibatch's expert segments (args.mb_off / mb_toff:
// row offsets and chunk prefixes per minibatch, args.mb_start: the tiles before each minibatch),
// wait for a minibatch's rows before loading them, and count each tile's epilogue warps out on
// args.consumed so that the slot can be refilled.  Once a gathering pair has gathered its share of
// every minibatch it runs tiles too.  So the tiles are not dealt in a fixed order but taken from
// one counter (args.ticket) in tile order: the even CTA's producer takes a tile and passes it to
// the roles of both CTAs through a TQ-deep queue in shared memory (each entry with a full
// barrier in both CTAs and an empty barrier in the even CTA); -1 ends the queue.  Which pair
// computes a tile does not change its result: each output element is still one tile's
// accumulator over K in a fixed order.
// MODE of narrow_body: the fixed deal over the whole layer (pair p takes tiles p, p + npairs, ...),
// the same tiles taken from a counter through the tile queue (NARROW_PLAIN_TICKET: a pair whose
// SMs run slower, or whose tiles cost more, takes fewer), the ring forward's GEMM1 (tiles from a
// ticket, each minibatch's rows awaited in the token ring) or, in the persistent ring forward,
// its GEMM2 (tiles from a second ticket, each minibatch's rows of a awaited from GEMM1).
constexpr int NARROW_PLAIN = 0, NARROW_RING_GEMM1 = 1, NARROW_RING_GEMM2 = 2, NARROW_PLAIN_TICKET = 3;
constexpr uint32_t kTmemOwn = 0xffffffffu;  // narrow_body allocates (and frees) its own TMEM

// One narrow-segment grouped GEMM on the CTA pairs of the launch.  `smem` is the CTA's 1024-byte
// aligned dynamic shared memory; tmem_given is a TMEM base allocated by the caller for both CTAs
// of the pair (at least C::TMEM_COLS columns), or kTmemOwn.  With a caller's TMEM the shared memory
// is left for another phase: the barriers are invalidated before returning.
template <bool WMN, bool SPLIT, int NMAX, int EPI, int MODE>
__device__ __forceinline__ void narrow_body(const CUtensorMap& tmW, const CUtensorMap& tmX, const CUtensorMap& tmX2,
                                            const CUtensorMap& tmXs, const CUtensorMap& tmX2s,
                                            const GemmArgs& args, uint8_t* smem, uint32_t tmem_given) {
  using C = NarrowCfg<WMN, SPLIT, NMAX, EPI>;
  constexpr bool RING = MODE == NARROW_RING_GEMM1 || MODE == NARROW_RING_GEMM2;
  constexpr bool QUEUE = MODE != NARROW_PLAIN;  // tiles from args.ticket through the tile queue
  constexpr int STAGES = C::STAGES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  float* xbuf = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);  // C::XBUF_BYTES
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + C::XBUF_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, tq_full[TQ], tq_empty[TQ], then
  // the TMEM address and the abort flag; at +C::QOFF the tile queue's entries (QUEUE)
  constexpr int TQ = C::TQ;
  static_assert((2 * STAGES + 5 + 2 * TQ) * 8 + 8 <= C::QOFF && C::QOFF + TQ * NARROW_QE * 4 <= C::BAR_BYTES,
                "barriers, TMEM address, abort flag and tile queue");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5 + 2 * TQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* tq = reinterpret_cast<volatile int*>(reinterpret_cast<uint8_t*>(bars) + C::QOFF);
  int* s_off = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + C::XBUF_BYTES + C::BAR_BYTES);
  typename C::coff_t* s_coff = reinterpret_cast<typename C::coff_t*>(s_off + (args.E + 1));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
  const int pair = (int)blockIdx.x >> 1;  // the fixed deal (not QUEUE)
  const int npairs = (int)gridDim.x >> 1;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + 2 + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * STAGES + 4]);
  auto tq_full = [&](int q) { return smem_u32(&bars[2 * STAGES + 5 + q]); };
  auto tq_empty = [&](int q) { return smem_u32(&bars[2 * STAGES + 5 + TQ + q]); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * C::EPI_WARPS);  // every epilogue warp of both CTAs
    }
    for (int q = 0; q < TQ; ++q) {
      mbar_init(tq_full(q), 1);
      // readers of a queue entry: the even CTA's MMA warp and the odd CTA's producer, and every
      // epilogue warp of both CTAs
      mbar_init(tq_empty(q), 2 + 2 * C::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // the whole layer's segments and chunk prefixes (RING decodes through the minibatch tables)
  if (!RING)
    for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_off[i] = args.offsets[i];
  __syncthreads();
  if (!RING && threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < args.E; ++e) {
      s_coff[e] = (typename C::coff_t)acc;
      acc += (s_off[e + 1] - s_off[e] + C::NMAX - 1) / C::NMAX;
    }
    s_coff[args.E] = (typename C::coff_t)acc;
  }
  if (warp == 1 && tmem_given == kTmemOwn) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem_base = tmem_given == kTmemOwn ? *tmem_slot : tmem_given;

  const int MT = C::m_tiles(args);
  // GEMM2 of the ring forward: the minibatch tables count GEMM1 tiles (args.mb_tiles1 per row
  // chunk); the same row chunks give MT GEMM2 tiles each
  auto tiles_before = [&](int mb) {
    return MODE == NARROW_RING_GEMM2 ? args.mb_start[mb] / args.mb_tiles1 * MT : args.mb_start[mb];
  };
  const int total = RING ? tiles_before(args.n_mb) : (int)s_coff[args.E] * MT;
  const int nkb = args.K / BK;
  // Tile g.  RING: the minibatch mb holding it, the tile decoded inside it, its rows' position in the
  // ring (ring_row0) and its rows' position in the outputs (t.row0, all rows of the layer).
  auto decode = [&](int g, int& mb, int& ring_row0) -> NarrowTile {
    if (!RING) {
      mb = 0;
      const NarrowTile t = decode_narrow_tile(g, MT, args.E, C::NMAX, s_off, s_coff);
      ring_row0 = t.row0;
      return t;
    }
    int lo = 0, hi = args.n_mb;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tiles_before(mid) <= g) lo = mid; else hi = mid;
    }
    mb = lo;
    NarrowTile t = decode_narrow_tile(g - tiles_before(lo), MT, args.E, C::NMAX,
                                      args.mb_off + (size_t)lo * (args.E + 1), args.mb_toff + (size_t)lo * (args.E + 1));
    ring_row0 = ((lo + args.ring_shift) % args.ring_slots) * args.mb_rows + t.row0;
    t.row0 += lo * args.mb_rows;
    if (MODE == NARROW_RING_GEMM2) ring_row0 = t.row0;  // a is read from the layer's rows
    return t;
  };

  // QUEUE: the n-th tile of this pair, from the tile queue (g = -1: no more).  The even CTA's
  // producer (one thread) takes each tile from the ticket counter (g_taken: the atomic is issued a
  // few K blocks before the tile is published, so that its round trip overlaps the loads), decodes
  // it once (the minibatch tables are in global memory: a binary search over the minibatches and
  // one over the experts) and writes the decoded tile into entry n % TQ of both CTAs' queues, one
  // tile ahead of its own loads; every other reader waits for the entry, reads it and counts
  // itself out on the even CTA's empty barrier of the entry.
  auto publish_tile = [&](int n, int g_taken, int& g, NarrowTile& t, int& mb, int& rr) -> bool {
    const int q = n % TQ;
    const uint32_t u = (uint32_t)(n / TQ) & 1u;
    if (!mbar_wait<true>(tq_empty(q), u ^ 1, abort_flag, args.status, SITE_RING_WAIT, kWaitLimitNs, 32))
      return false;
    g = g_taken < total ? g_taken : -1;
    if (g >= 0) t = decode(g, mb, rr);
    const int v[10] = {g, t.e, t.c, t.m, t.nc, t.row0, t.rows, t.n, mb, rr};
    volatile int* dst = tq + q * NARROW_QE;
    const uint32_t peer = mapa_shared(smem_u32(const_cast<int*>(dst)), 1);
#pragma unroll
    for (int i = 0; i < 10; ++i) {
      dst[i] = v[i];
      st_shared_cluster_u32(peer + 4u * i, (uint32_t)v[i]);
    }
    mbar_arrive(tq_full(q));
    mbar_arrive_cluster(mapa_shared(tq_full(q), 1));  // release: the peer's copy is written
    return true;
  };
  // by all lanes of a warp (lane 0 waits and counts out) or by a single thread (warp_wide false)
  auto read_tile = [&](int n, int& g, NarrowTile& t, int& mb, int& rr, uint32_t sleep_ns, bool warp_wide) -> bool {
    const int q = n % TQ;
    const uint32_t u = (uint32_t)(n / TQ) & 1u;
    int w_ok = 1;
    if (lane == 0 || !warp_wide)
      w_ok = mbar_wait<true>(tq_full(q), u, abort_flag, args.status, SITE_RING_WAIT, kWaitLimitNs, sleep_ns);
    if (warp_wide) {
      w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      __syncwarp();
    }
    if (!w_ok) return false;
    const volatile int* src = tq + q * NARROW_QE;
    g = src[0];
    t.e = src[1];
    t.c = src[2];
    t.m = src[3];
    t.nc = src[4];
    t.row0 = src[5];
    t.rows = src[6];
    t.n = src[7];
    mb = src[8];
    rr = src[9];
    if (warp_wide) __syncwarp();  // every lane has read the entry
    if (lane == 0 || !warp_wide) {
      if (rank == 0) mbar_arrive(tq_empty(q));
      else mbar_arrive_cluster(mapa_shared(tq_empty(q), 0));
    }
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmXs);
      if (SPLIT) {
        tma_prefetch_desc(&tmX2);
        tma_prefetch_desc(&tmX2s);
      }
      const uint64_t pol_rows = l2_policy_evict_last();   // rows: read by every weight tile
      const uint64_t pol_once = l2_policy_evict_first();  // a weight tile read by one chunk
      const uint64_t pol_shared = l2_policy_evict_normal();
      const uint32_t full0_cl = mapa_shared(full_bar(0), 0);  // the even CTA's full barriers
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      int ring_ready = -1;  // RING: last minibatch known to be ready (gathered, or through GEMM1)
      // QUEUE, even CTA: the tile after the current one is taken during the current one's loads
      int g_nx = 0, mb_nx = 0, rr_nx = 0;
      NarrowTile t_nx{};
      bool have_nx = false;
      if (QUEUE && rank == 0) {
        ok = publish_tile(0, atomicAdd(args.ticket, 1), g_nx, t_nx, mb_nx, rr_nx);
        have_nx = true;
      }
      for (int n = 0; ok; ++n) {
        int g, mb = 0, ring_row0 = 0;
        NarrowTile t{};
        if (!QUEUE) {
          g = pair + n * npairs;
          if (g >= total) break;
          t = decode(g, mb, ring_row0);
        } else if (rank == 0) {
          g = g_nx;
          t = t_nx;
          mb = mb_nx;
          ring_row0 = rr_nx;
          have_nx = false;
        } else if (!read_tile(n, g, t, mb, ring_row0, 32, false)) {
          ok = false;
          break;
        }
        if (g < 0) break;
        if (RING && mb > ring_ready) {
          // GEMM1: the minibatch's rows must be in the ring before the first load of its tiles;
          // GEMM2: every GEMM1 tile of the minibatch must have stored its rows of a
          const bool ready =
              MODE == NARROW_RING_GEMM1
                  ? wait_counter(&args.gathered[mb], min(args.mb_rows, args.R - mb * args.mb_rows), args.status,
                                 SITE_RING_WAIT)
                  : wait_counter(&args.consumed[mb], args.consume_per_tile * (args.mb_start[mb + 1] - args.mb_start[mb]),
                                 args.status, SITE_RING_WAIT);
          if (!ready) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          fence_proxy_async_global();
          ring_ready = mb;
        }
        const int half = t.n >> 1;                      // rows of this CTA's half of N
        int n64;
        bool with32;
        const int xrows = narrow_x_boxes(half, n64, with32);  // <= NMAX / 2: fits the X buffer
        const int x_row = ring_row0 + (int)rank * half;
        const int w_row = t.m * C::PM + 128 * (int)rank;
        const uint32_t pair_tx = 2u * (C::A_BYTES + C::X_OPS * xrows * 128);
        const uint64_t pol_w = t.nc > 1 ? pol_shared : pol_once;
        const int kb_pub = nkb - 1 < STAGES ? nkb - 1 : STAGES;  // the stage ring is full by then
        int g_taken = 0;
        for (int kb = 0; kb < nkb; ++kb) {
          if (QUEUE && rank == 0 && !have_nx && kb == 0) g_taken = atomicAdd(args.ticket, 1);
          if (QUEUE && rank == 0 && !have_nx && kb == kb_pub) {
            if (!publish_tile(n + 1, g_taken, g_nx, t_nx, mb_nx, rr_nx)) {
              ok = false;
              break;
            }
            have_nx = true;
          }
          if (!mbar_wait<true>(empty_bar(stage), phase ^ 1, abort_flag, args.status, SITE_GEMM_PRODUCER_EMPTY,
                               kWaitLimitNs, 32)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0_cl + 8u * stage;
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sx = sa + C::A_BYTES;
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), pair_tx);
          const int k0 = kb * BK;
          if (EPI == EPI_SWIGLU) {
            // 64 gate rows, then the 64 up rows of the same intermediate indices
            tma_load_4d_pair(sa, &tmW, fb, k0, t.m * 128 + 64 * (int)rank, 0, t.e, pol_w);
          } else if (EPI == EPI_SWIGLU_PAIRED) {
            // 128 gate rows, then the 128 up rows of the same intermediate indices
            tma_load_4d_pair(sa, &tmW, fb, k0, t.m * 256 + 128 * (int)rank, 0, t.e, pol_w);
          } else if (EPI == EPI_F32_PAIRED) {
            // this CTA's 128 rows of each of the two weight tiles of a 512-row pair tile
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int wr = t.m * 2 * C::PM + h * C::PM + 128 * (int)rank;
              const uint32_t sh = sa + h * (C::A_BYTES / 2);
              if (WMN) {
                tma_load_3d_pair(sh, &tmW, fb, wr, k0, t.e, pol_w);
                tma_load_3d_pair(sh + MN_ATOM_BYTES, &tmW, fb, wr + 64, k0, t.e, pol_w);
              } else {
                tma_load_3d_pair(sh, &tmW, fb, k0, wr, t.e, pol_w);
              }
            }
          } else if (WMN) {
            tma_load_3d_pair(sa, &tmW, fb, w_row, k0, t.e, pol_w);
            tma_load_3d_pair(sa + MN_ATOM_BYTES, &tmW, fb, w_row + 64, k0, t.e, pol_w);
          } else {
            tma_load_3d_pair(sa, &tmW, fb, k0, w_row, t.e, pol_w);
          }
          for (int b = 0; b < n64; ++b) {
            const int r = b * NARROW_XBOX;
            tma_load_2d_pair(sx + r * 128, &tmX, fb, k0, x_row + r, pol_rows);
            if (SPLIT) tma_load_2d_pair(sx + C::X_OP + r * 128, &tmX2, fb, k0, x_row + r, pol_rows);
          }
          if (with32) {
            const int r = n64 * NARROW_XBOX;
            tma_load_2d_pair(sx + r * 128, &tmXs, fb, k0, x_row + r, pol_rows);
            if (SPLIT) tma_load_2d_pair(sx + C::X_OP + r * 128, &tmX2s, fb, k0, x_row + r, pol_rows);
          }
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
      const uint32_t a_lbo = WMN ? MOK_MN_LBO : 16, a_sbo = WMN ? MOK_MN_SBO : 1024;
      for (int n = 0; ok; ++n) {
        int g, mb_unused = 0, rr_unused = 0;
        NarrowTile t{};
        if (QUEUE) {
          if (!read_tile(n, g, t, mb_unused, rr_unused, 32, true)) {
            ok = false;
            break;
          }
        } else {
          g = pair + n * npairs;
          if (g >= total) break;
          t = decode(g, mb_unused, rr_unused);
        }
        if (g < 0) break;
        uint32_t idesc = idesc_bf16_f32(C::PM, t.n, WMN, false);
        if (args.f16) idesc &= ~((1u << 7) | (1u << 10));  // A and B formats: fp16 instead of bf16
        int w_ok = 1;
        if (lane == 0)
          w_ok = mbar_wait<true>(tempty_bar(acc), acc_phase ^ 1, abort_flag, args.status, SITE_GEMM_MMA_TMEM_EMPTY);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::NMAX;  // paired: acc = 0, up rows at +256
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
            const uint32_t sx = sa + C::A_BYTES;
#pragma unroll
            for (int k16 = 0; k16 < BK / 16; ++k16) {
              const uint64_t adesc = smem_desc_sw128(sa + (WMN ? k16 * 2048 : k16 * 32), a_lbo, a_sbo);
              const uint64_t bdesc = smem_desc_sw128(sx + k16 * 32, 16, 1024);
              const uint32_t first = (kb | k16) != 0 ? 1u : 0u;
              umma_f16_pair(d_tmem, adesc, bdesc, idesc, first);
              if (SPLIT) umma_f16_pair(d_tmem, adesc, smem_desc_sw128(sx + C::X_OP + k16 * 32, 16, 1024), idesc, 1u);
              if (C::kPaired) {
                // the second weight tile (or the up rows): the other half of this stage's A
                const uint64_t adesc2 =
                    smem_desc_sw128(sa + C::A_BYTES / 2 + (WMN ? k16 * 2048 : k16 * 32), a_lbo, a_sbo);
                umma_f16_pair(d_tmem + 256, adesc2, bdesc, idesc, first);
                if (SPLIT)
                  umma_f16_pair(d_tmem + 256, adesc2, smem_desc_sw128(sx + C::X_OP + k16 * 32, 16, 1024), idesc, 1u);
              }
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
        acc = (acc + 1) % C::ACCS;
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
  } else if (warp < 2 + C::EPI_WARPS) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 are reachable by this warp
    const uint32_t tempty0_cl = mapa_shared(tempty_bar(0), 0);
    float* out = reinterpret_cast<float*>(args.out0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int n = 0;; ++n) {
      int g, mb = 0, rr_unused = 0;
      NarrowTile t{};
      if (QUEUE) {
        if (!read_tile(n, g, t, mb, rr_unused, 256, true)) break;
      } else {
        g = pair + n * npairs;
        if (g >= total) break;
        t = decode(g, mb, rr_unused);
      }
      if (g < 0) break;
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait<true>(tfull_bar(acc), acc_phase, abort_flag, args.status, SITE_GEMM_EPI_TMEM_FULL,
                               kWaitLimitNs, 256);
      const uint32_t tacc = tmem_base + acc * C::NMAX + (uint32_t(quarter * 32) << 16);
      if (EPI == EPI_SWIGLU) {
        // the two warps that share intermediate indices agree on stopping (one of them may
        // have given up waiting while the other saw the accumulator complete)
        const int qp = quarter & 1;
        const bool w_fail = !__shfl_sync(0xffffffffu, w_ok, 0);
        if (named_bar_any(1 + qp, 64, w_fail)) break;
        tc_fence_after();
        const bool gate = quarter < 2;  // lanes of gate rows (h); quarter + 2 holds u
        const int i = t.m * 128 + 64 * (int)rank + 32 * qp + lane;
        float* hu = reinterpret_cast<float*>(args.out0) + (long long)t.row0 * args.ld0;
        __nv_bfloat16* ahi = reinterpret_cast<__nv_bfloat16*>(args.out1) + (long long)t.row0 * args.ld1;
        __nv_bfloat16* alo = reinterpret_cast<__nv_bfloat16*>(args.out2) + (long long)t.row0 * args.ld1;
        float* xh = xbuf + qp * 2 * 32 * 32;  // [32 rows][32 lanes]: h, then u
        float* xu = xh + 32 * 32;
#pragma unroll 1
        for (int c = 0; c * 32 < t.rows; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tacc + c * 32, v);
          tmem_wait_ld();
          const int nr = min(32, t.rows - c * 32);
          const long long rb = c * 32;
          // both warps park their block in shared memory ([row][lane]: conflict-free), so the up
          // warp's SwiGLU loop needs no fully unrolled register block
          float* mine = gate ? xh : xu;
#pragma unroll
          for (int j = 0; j < 32; ++j) mine[j * 32 + lane] = __uint_as_float(v[j]);
          if (gate) {
            float* hp = hu + rb * args.ld0 + i;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (j < nr) *hp = __uint_as_float(v[j]);
              hp += args.ld0;
            }
          }
          named_bar_sync(1 + qp, 64);  // h of this block is in shared memory
          if (!gate) {
            float* up = hu + rb * args.ld0 + args.I + i;
            __nv_bfloat16* php = ahi + rb * args.ld1 + i;
            __nv_bfloat16* plp = alo + rb * args.ld1 + i;
#pragma unroll 4
            for (int j = 0; j < nr; ++j) {
              const float h = xh[j * 32 + lane];
              const float u = xu[j * 32 + lane];
              *up = u;
              const float a = h / (1.0f + __expf(-h)) * u;
              if (args.a_f16) {
                *reinterpret_cast<__half*>(php) = __float2half_rn(a);
              } else {
                const __nv_bfloat16 a_hi = __float2bfloat16_rn(a);
                *php = a_hi;
                *plp = __float2bfloat16_rn(a - __bfloat162float(a_hi));
              }
              up += args.ld0;
              php += args.ld1;
              plp += args.ld1;
            }
          }
          named_bar_sync(1 + qp, 64);  // the up warp has read it
        }
      } else if (EPI == EPI_SWIGLU_PAIRED) {
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
        tc_fence_after();
        // this thread's intermediate index: h in column n, u in column 256 + n of its lane; the
        // warp's group takes every other 8-row block
        const int i = t.m * 256 + 128 * (int)rank + 32 * quarter + lane;
        const int grp = (warp - 2) >> 2;
        float* hrow = reinterpret_cast<float*>(args.out0) + (long long)t.row0 * args.ld0 + i;
        __nv_bfloat16* arow_hi = reinterpret_cast<__nv_bfloat16*>(args.out1) + (long long)t.row0 * args.ld1 + i;
        __nv_bfloat16* arow_lo = reinterpret_cast<__nv_bfloat16*>(args.out2) + (long long)t.row0 * args.ld1 + i;
#pragma unroll 1
        for (int n0 = 8 * grp; n0 < t.rows; n0 += 8 * (C::EPI_WARPS / 4)) {
          uint32_t hv[8], uv[8];
          tmem_ld_32x32b_x8(tacc + n0, hv);
          tmem_ld_32x32b_x8(tacc + 256 + n0, uv);
          tmem_wait_ld();
          const int nr = min(8, t.rows - n0);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j < nr) {
              const float h = __uint_as_float(hv[j]);
              const float u = __uint_as_float(uv[j]);
              const long long r = n0 + j;
              hrow[r * args.ld0] = h;
              hrow[r * args.ld0 + args.I] = u;
              const float a = h / (1.0f + __expf(-h)) * u;
              if (args.a_f16) {
                reinterpret_cast<__half*>(arow_hi)[r * args.ld1] = __float2half_rn(a);
              } else {
                const __nv_bfloat16 a_hi = __float2bfloat16_rn(a);
                arow_hi[r * args.ld1] = a_hi;
                arow_lo[r * args.ld1] = __float2bfloat16_rn(a - __bfloat162float(a_hi));
              }
            }
          }
        }
      } else {
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
        tc_fence_after();
        // this thread's output column; the accumulator's columns are the chunk's rows (paired:
        // the second weight tile, 256 output columns further, in accumulator columns 256 + n)
#pragma unroll 1
        for (int half = 0; half < (C::kPaired ? 2 : 1); ++half) {
          const int j = t.m * (C::kPaired ? 2 : 1) * C::PM + half * C::PM + 128 * (int)rank + 32 * quarter + lane;
          const bool jv = j < args.N;
          float* o = out + (long long)t.row0 * args.ld0 + j;
          const uint32_t th = tacc + half * 256;
#pragma unroll 1
          for (int c = 0; c * 32 < t.rows; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(th + c * 32, v);
            tmem_wait_ld();
            const int nr = min(32, t.rows - c * 32);
            if (jv) {
              float* oc = o + (long long)(c * 32) * args.ld0;
              if (nr == 32) {
#pragma unroll
                for (int i = 0; i < 32; ++i) oc[(long long)i * args.ld0] = __uint_as_float(v[i]);
              } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (i < nr) oc[(long long)i * args.ld0] = __uint_as_float(v[i]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty0_cl + 8u * acc);
      // GEMM1 of the ring: this warp is done with the tile (its MMAs have read the rows): once
      // every epilogue warp of every tile of the minibatch has counted in, its ring slot may be
      // refilled (and, with args.fence_out, GEMM2 may read the minibatch's rows of a).  GEMM2 of
      // the persistent ring forward: the warp's rows of o are stored (args.done, for the combine).
      if (RING) {
        if (MODE == NARROW_RING_GEMM2 || args.fence_out) {
          __threadfence();  // this lane's stores, before the count (release, with the warp sync)
          __syncwarp();
        }
        if (lane == 0) atomicAdd(MODE == NARROW_RING_GEMM2 ? args.done : &args.consumed[mb], 1);
      }
      acc = (acc + 1) % C::ACCS;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or signals may still touch it
  if (tmem_given == kTmemOwn) {
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
  } else {
    // another phase sets up its barriers in this shared memory next
    if (threadIdx.x == 0)
      for (int i = 0; i < 2 * STAGES + 5 + 2 * TQ; ++i)
        mbar_inval(smem_u32(&bars[i]));
    __syncthreads();
  }
}

template <bool WMN, bool SPLIT, int NMAX, int EPI, int KMODE = NARROW_PLAIN>
__global__ void __launch_bounds__(NarrowCfg<WMN, SPLIT, NMAX, EPI>::THREADS, 1)
    gemm_narrow_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmXs,
                       const __grid_constant__ CUtensorMap tmX2s, const GemmArgs args) {
  using C = NarrowCfg<WMN, SPLIT, NMAX, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (KMODE == NARROW_RING_GEMM1) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::XBUF_BYTES);
    ring_gather_first(args);
    if ((int)blockIdx.x < args.comm_ctas) {
      ring_gather(args, smem, C::STAGES * C::STAGE_BYTES, bars);
      ring_gather_retire(args, C::STAGES * C::STAGE_BYTES, bars);  // then this pair runs tiles as well
    }
  }
  narrow_body<WMN, SPLIT, NMAX, EPI, KMODE>(tmW, tmX, tmX2, tmXs, tmX2s, args, smem, kTmemOwn);
}

// ------------------------------------------------------------------ persistent ring forward
//
// The whole ring forward after the schedule table in one cooperative launch, as the pages' two SM
// groups ("把 MoE 通信延迟从 103μs 压到 18μs：Cursor 开源 GPU 内核 MoK", aientropygate.com, §03 ②:
// one group runs dispatch, combine and state, the other the expert FFN, signalling through
// counters): every CTA copies minibatch 0; args1.comm_ctas CTAs gather the later minibatches into
// the token ring; the CTA pairs run GEMM1 + SwiGLU on each gathered minibatch (tiles from one
// ticket); then GEMM2 on each minibatch whose GEMM1 tiles have all stored their rows of a (tiles
// from a second ticket, so a pair takes GEMM2 tiles while others still finish GEMM1); then, once
// every GEMM2 tile has stored its rows of o, every warp of the launch takes tokens of the weighted
// merge.  The gathering CTAs join each stage once their gathering is done.  Each output element is
// computed as by the separate launches (same tiles, K order, epilogues and merge), so y is bitwise
// the same.
struct RingCombineArgs {
  const float* o;          // fp32 [R][H] expert outputs (written by this launch's GEMM2)
  const float* gates;      // f32 [T][k]
  const int32_t* row_of;   // i32 [T*k]
  int T, k, vec_per_row;   // vec_per_row = H / 8
  __nv_bfloat16* y;        // bf16 [T][H]
};

template <int EPI1, int EPI2>
struct RingFwdCfg {
  using C1 = NarrowCfg<false, false, 256, EPI1>;
  using C2 = NarrowCfg<false, true, 256, EPI2>;
  static_assert(!C1::kDeep && !C2::kDeep, "the phases share the standard barrier layout");
  static constexpr int THREADS = C1::THREADS > C2::THREADS ? C1::THREADS : C2::THREADS;
  // bytes each phase uses past the 1024-byte aligned base (stages, exchange buffer, barriers,
  // segment tables); the TMEM address follows the larger
  static __host__ __device__ constexpr int phase_end(int stages, int stage_bytes, int xbuf, int E) {
    return stages * stage_bytes + xbuf + NARROW_BAR_BYTES + 2 * (E + 1) * 4;  // C1, C2: not the deep form
  }
  static __host__ __device__ constexpr int tmem_slot_offset(int E) {
    return phase_end(C1::STAGES, C1::STAGE_BYTES, C1::XBUF_BYTES, E) >
                   phase_end(C2::STAGES, C2::STAGE_BYTES, C2::XBUF_BYTES, E)
               ? phase_end(C1::STAGES, C1::STAGE_BYTES, C1::XBUF_BYTES, E)
               : phase_end(C2::STAGES, C2::STAGE_BYTES, C2::XBUF_BYTES, E);
  }
  // TMEM address (16 bytes), then the merge's two barriers (16 bytes)
  static __host__ __device__ constexpr size_t smem_bytes(int E) { return 1024 + size_t(tmem_slot_offset(E)) + 32; }
  // the merge: a token's k <= 8 rows of o in parts of at most MERGE_VEC 8-column groups, two
  // buffers of 8 row parts each (96 KB), refilled by bulk copies
  static constexpr int MERGE_VEC = 192;
  static_assert(2 * 8 * MERGE_VEC * 32 <= C1::STAGES * C1::STAGE_BYTES, "merge buffers in the stage memory");
  static_assert(C1::TMEM_COLS <= 512 && C2::TMEM_COLS <= 512, "both GEMMs fit one TMEM allocation");
};

template <int EPI1, int EPI2>
__global__ void __launch_bounds__(RingFwdCfg<EPI1, EPI2>::THREADS, 1)
    ring_forward_kernel(const __grid_constant__ CUtensorMap tm1W, const __grid_constant__ CUtensorMap tm1X,
                        const __grid_constant__ CUtensorMap tm1Xs, const __grid_constant__ CUtensorMap tm2W,
                        const __grid_constant__ CUtensorMap tm2X, const __grid_constant__ CUtensorMap tm2X2,
                        const __grid_constant__ CUtensorMap tm2Xs, const __grid_constant__ CUtensorMap tm2X2s,
                        const GemmArgs a1, const GemmArgs a2, const RingCombineArgs cb) {
  using R = RingFwdCfg<EPI1, EPI2>;
  using C1 = typename R::C1;
  using C2 = typename R::C2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + R::tmem_slot_offset(a1.E));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  ring_gather_first(a1);
  if ((int)blockIdx.x < a1.comm_ctas) {
    uint64_t* gbars = reinterpret_cast<uint64_t*>(smem + C1::STAGES * C1::STAGE_BYTES + C1::XBUF_BYTES);
    ring_gather(a1, smem, C1::STAGES * C1::STAGE_BYTES, gbars);
    ring_gather_retire(a1, C1::STAGES * C1::STAGE_BYTES, gbars);  // then this pair runs tiles as well
  }
  // one TMEM allocation of both CTAs of the pair for the two GEMMs
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  narrow_body<false, false, 256, EPI1, NARROW_RING_GEMM1>(tm1W, tm1X, tm1X, tm1Xs, tm1Xs, a1, smem, tmem_base);
  narrow_body<false, true, 256, EPI2, NARROW_RING_GEMM2>(tm2W, tm2X, tm2X2, tm2Xs, tm2X2s, a2, smem, tmem_base);

  // The weighted merge, once every GEMM2 epilogue warp of every tile has counted out.  Items are
  // (token, part of its columns); the CTA's warp 0 bulk-copies an item's k row parts of o into
  // one of two shared-memory buffers while every thread merges the other, so that each SM keeps
  // up to 96 KB of o in flight (a warp per token, as the merge kernel, kept too little in flight
  // with one CTA per SM here).  Per output the same fp32 sum over j = 0..k-1 and one rounding.
  const int total2 = a2.mb_start[a2.n_mb] / a2.mb_tiles1 * C2::m_tiles(a2);
  uint64_t* mbars = reinterpret_cast<uint64_t*>(smem + R::tmem_slot_offset(a1.E) + 16);
  int ok = 1;
  if (threadIdx.x == 0) {
    ok = wait_counter(a2.done, 2 * C2::EPI_WARPS * total2, a2.status, SITE_RING_WAIT);
    mbar_init(smem_u32(&mbars[0]), 1);
    mbar_init(smem_u32(&mbars[1]), 1);
    fence_mbar_init();
    fence_proxy_async_global();  // o, stored by other CTAs, is read by bulk copies
  }
  if (!__syncthreads_or(!ok)) {
    constexpr int MV = R::MERGE_VEC;
    const int parts = (cb.vec_per_row + MV - 1) / MV;
    const int items = cb.T * parts;
    auto part_vec = [&](int part) { return min(MV, cb.vec_per_row - part * MV); };
    auto buf = [&](int b, int j) { return smem + (size_t)(b * 8 + j) * MV * 32; };
    auto issue = [&](int item, int b) {  // warp 0: lane j copies row part j
      const int t = item / parts, part = item - t * parts;
      const uint32_t bytes = (uint32_t)part_vec(part) * 32;
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(&mbars[b]), bytes * cb.k);
      __syncwarp();
      if (lane < cb.k) {
        const int row = cb.row_of[(size_t)t * cb.k + lane];
        bulk_load_g2s(smem_u32(buf(b, lane)), cb.o + (size_t)row * cb.vec_per_row * 8 + (size_t)part * MV * 8,
                      bytes, smem_u32(&mbars[b]));
      }
    };
    if (warp == 0 && (int)blockIdx.x < items) issue(blockIdx.x, 0);
    bool live = true;
    for (int i = 0; live; ++i) {
      const int item = (int)blockIdx.x + i * (int)gridDim.x;
      if (item >= items) break;
      const int b = i & 1;
      // the other buffer was merged in the previous iteration (all threads passed its barrier)
      if (warp == 0 && item + (int)gridDim.x < items) issue(item + (int)gridDim.x, b ^ 1);
      const int t = item / parts, part = item - t * parts;
      float wj[8];  // loaded while the row parts land
#pragma unroll
      for (int j = 0; j < 8; ++j) wj[j] = j < cb.k ? cb.gates[(size_t)t * cb.k + j] : 0.0f;
      volatile int no_abort = 0;
      live = mbar_wait(smem_u32(&mbars[b]), (uint32_t)(i >> 1) & 1u, &no_abort, a2.status, SITE_RING_WAIT);
      if (live) {
        const int pv = part_vec(part);
        for (int v = threadIdx.x; v < pv; v += blockDim.x) {
          float acc[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < cb.k) {
              const uint4* p = reinterpret_cast<const uint4*>(buf(b, j)) + 2 * v;
              acc_f32x8(acc, p[0], p[1], wj[j]);
            }
          reinterpret_cast<uint4*>(cb.y)[(size_t)t * cb.vec_per_row + (size_t)part * MV + v] = pack_bf16x8(acc);
        }
      }
      live = !__syncthreads_or(!live);
    }
    if (threadIdx.x == 0) {
      mbar_inval(smem_u32(&mbars[0]));
      mbar_inval(smem_u32(&mbars[1]));
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

}  // namespace mok
