// Host launchers of the tcgen05 GEMMs: TMA descriptor encoding and the kernel
// instantiations used by the forward and backward of the layer.
#include <cuda.h>

#include <mutex>

#include "gemm.cuh"
#include "gemm_narrow.cuh"
#include "gemm_pair.cuh"
#include "wgrad.cuh"
#include "wgrad_pair.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace mok {

namespace {

// out_map / out1 / out2: store maps of the outputs for epilogues that use TMA stores.
template <int MODE, int EPI, int SPLIT, int BN>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b, const CUtensorMap& b2,
                   const GemmArgs& args, int grid, cudaStream_t st, const CUtensorMap* out_map = nullptr,
                   const CUtensorMap* out1 = nullptr, const CUtensorMap* out2 = nullptr) {
  using C = GemmCfg<MODE, EPI, SPLIT, BN>;
  static_assert(C::smem_bytes(1024) <= 232448, "shared memory budget");
  if (grid <= 0) return cudaSuccess;
  auto kern = gemm_kernel<MODE, EPI, SPLIT, BN>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem_bytes(1024));
  if (err != cudaSuccess) return err;
  if (C::kTmaEpi && out_map == nullptr) return cudaErrorInvalidValue;
  if (EPI == EPI_SWIGLU && C::kTmaEpi && (out1 == nullptr || out2 == nullptr)) return cudaErrorInvalidValue;
  kern<<<grid, C::THREADS, C::smem_bytes(args.E), st>>>(a, a2, b, b2, out_map ? *out_map : a, out1 ? *out1 : a,
                                                        out2 ? *out2 : a, args);
  return cudaGetLastError();
}


// Upper bound of the 128-row tiles of R expert-sorted rows split into E segments.
int row_tiles_bound(int R, int E) { return (R + BM - 1) / BM + E; }

// CTA-pair GEMM: clusters of 2 CTAs, one pair per two SMs (as many as can be co-resident).
template <int EPI, int SPLIT>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b, const CUtensorMap& o0,
                        const CUtensorMap& o1, const CUtensorMap& o2, const GemmArgs& args, int pair_tiles_bound,
                        int n_sm, cudaStream_t st) {
  using C = PairCfg<EPI, SPLIT>;
  static_assert(C::smem_bytes(1024) <= 232448, "shared memory budget");
  if (pair_tiles_bound <= 0) return cudaSuccess;
  auto kern = gemm_pair_kernel<EPI, SPLIT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem_bytes(1024));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::smem_bytes(args.E);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // co-resident pairs of this kernel on this device (cached per device)
  static int max_pairs[64] = {0};
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_pairs[dev] == 0) {
    cfg.gridDim = dim3(2 * std::max(1, n_sm / 2), 1, 1);
    int clusters = 0;
    if ((err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return err;
    max_pairs[dev] = std::max(1, clusters);
  }
  const int pairs = std::min(pair_tiles_bound, max_pairs[dev]);
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  err = cudaLaunchKernelEx(&cfg, kern, a, a2, b, o0, o1, o2, args);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// Upper bound of the 256-row pair tiles of R expert-sorted rows split into E segments (also of
// the narrow kernel's row chunks).
int pair_tiles_bound(int R, int E) { return (R + 255) / 256 + E; }

// Split-operand narrow GEMMs (GEMM2, dX_g): when experts average at most 160 rows, two 256-row
// weight tiles per pair tile sharing the row stages (EPI_F32_PAIRED: about 57% of each stage's
// bytes are weights instead of 40%, which these fill-bound GEMMs turn into weight bandwidth;
// measured at 128 rows per expert dX_g 3.02 -> 2.76 ms, GEMM2 1.58 -> 1.57 ms), in chunks of at
// most 256 rows (three stages either way; 192-row chunks cut the long experts of a skewed layer
// into more chunks, each of which streams the weight tiles again); else one weight tile (at 512
// rows per expert GEMM2 is near its MMA rate, where pairing gained nothing).

// Narrow-segment GEMM on CTA pairs: W (K-major [E][N][K] or, WMN, MN-major [E][K][N]) against
// expert-sorted rows X [R][K] (hi, and lo when SPLIT; x_lo is ignored otherwise); fp32 out
// [R][N] (row stride ld).
template <bool WMN, bool SPLIT, int NMAX, int EPI = EPI_F32>
cudaError_t launch_narrow(const CUtensorMap& w, const void* x_hi, const void* x_lo, int K, GemmArgs args, int R,
                          int n_sm, cudaStream_t st) {
  using C = NarrowCfg<WMN, SPLIT, NMAX, EPI>;
  static_assert(C::smem_bytes(C::kDeep ? NARROW_DEEP_MAX_E : 1024) <= 232448, "shared memory budget");
  if (C::kDeep && args.E > NARROW_DEEP_MAX_E) return cudaErrorInvalidValue;
  CUtensorMap tx, tx2, txs, tx2s;
  if (!tmap_2d(&tx, x_hi, K, R, BK, NARROW_XBOX) || !tmap_2d(&txs, x_hi, K, R, BK, NARROW_XBOX_S))
    return cudaErrorInvalidValue;
  tx2 = tx;
  tx2s = txs;
  if (SPLIT && (!tmap_2d(&tx2, x_lo, K, R, BK, NARROW_XBOX) || !tmap_2d(&tx2s, x_lo, K, R, BK, NARROW_XBOX_S)))
    return cudaErrorInvalidValue;
  const int bound = ((R + NMAX - 1) / NMAX + args.E) * C::m_tiles(args);
  if (R <= 0 || bound <= 0) return cudaSuccess;
  // tiles from a counter when the launch has one (args.ticket, zero at launch), else a fixed deal
  auto kern = args.ticket != nullptr ? gemm_narrow_kernel<WMN, SPLIT, NMAX, EPI, NARROW_PLAIN_TICKET>
                                     : gemm_narrow_kernel<WMN, SPLIT, NMAX, EPI, NARROW_PLAIN>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::smem_bytes(C::kDeep ? NARROW_DEEP_MAX_E : 1024));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::smem_bytes(args.E);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_pairs[2][64] = {};  // co-resident pairs of each kernel, per device
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int& mp = max_pairs[args.ticket != nullptr][dev];
  if (mp == 0) {
    cfg.gridDim = dim3(2 * std::max(1, n_sm / 2), 1, 1);
    int clusters = 0;
    if ((err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return err;
    mp = std::max(1, clusters);
  }
  cfg.gridDim = dim3(2 * std::min(bound, mp), 1, 1);
  err = cudaLaunchKernelEx(&cfg, kern, w, tx, tx2, txs, tx2s, args);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_gemm(const void* x, const void* w_router, int T, int H, int E, float* logits,
                               int* status, int n_sm, cudaStream_t st) {
  // A skinny GEMM (E columns, K = H).  With few token tiles (T = 4096: 32 tiles of 128 x 256 on
  // one SM in five, 56 us) 128 x 64 tiles spread it over four times the SMs, each A tile then read
  // four times (from L2: 47 us); with enough tiles for half the SMs the 128 x 256 tiles stay (at
  // T = 16384 the four reads of 235 MB of x no longer fit L2: 0.07 -> 0.18 ms)
  GemmArgs g = base_args(1, nullptr, nullptr, status);
  g.M = T;
  g.N = E;
  g.K = H;
  g.out0 = logits;
  g.ld0 = E;
  const int mt = (T + BM - 1) / BM;
  const bool narrow = mt * ((E + 255) / 256) < n_sm / 2;
  const int bn = narrow ? 64 : 256;
  CUtensorMap ta, tb;
  if (!tmap_2d(&ta, x, H, T, BK, BM) || !tmap_2d(&tb, w_router, H, E, BK, bn)) return cudaErrorInvalidValue;
  const int tiles = mt * ((E + bn - 1) / bn);
  g.total_tiles = tiles;
  if (narrow) return launch<MODE_DENSE, EPI_F32, SPLIT_NONE, 64>(ta, ta, tb, tb, g, std::min(tiles, n_sm), st);
  return launch<MODE_DENSE, EPI_F32, SPLIT_NONE, 256>(ta, ta, tb, tb, g, std::min(tiles, n_sm), st);
}

cudaError_t launch_gemm1_swiglu(const void* x_g, const void* w13, int R, int H, int I, int E,
                                const int32_t* offsets, const int32_t* tile_off, float* hu, void* act_hi,
                                void* act_lo, int* status, int n_sm, int variant, bool a_f16, cudaStream_t st) {
  if (a_f16 && variant != GEMM_NARROW) return cudaErrorInvalidValue;
  if (variant == GEMM_NARROW) {
    // W13[e] as [2][I][H]: each CTA takes 64 gate rows and their 64 up rows in one box (128 and
    // 128 in the paired form, at >= 384 rows per expert)
    const bool paired = (long long)R >= 384LL * E && I % 256 == 0;  // whole 256-index tiles
    CUtensorMap tw;
    if (!tmap_w13_gate_up(&tw, w13, H, I, E, paired ? 128 : 64)) return cudaErrorInvalidValue;
    GemmArgs g = base_args(E, offsets, tile_off, status);
    g.N = I;
    g.K = H;
    g.I = I;
    g.out0 = hu;
    g.ld0 = 2LL * I;
    g.out1 = act_hi;
    g.out2 = act_lo;
    g.ld1 = I;
    g.a_f16 = a_f16 ? 1 : 0;
    g.ticket = work_counter(status, CNT_GEMM1);
    if (paired) return launch_narrow<false, false, 256, EPI_SWIGLU_PAIRED>(tw, x_g, nullptr, H, g, R, n_sm, st);
    // at most 160 rows per expert on average: 192-row chunks (7 stages instead of 6; 1% faster at
    // 128 rows per expert)
    if (narrow_short_rows(R, E))
      return launch_narrow<false, false, 192, EPI_SWIGLU>(tw, x_g, nullptr, H, g, R, n_sm, st);
    return launch_narrow<false, false, 256, EPI_SWIGLU>(tw, x_g, nullptr, H, g, R, n_sm, st);
  }
  const bool pair = variant == GEMM_ROWS_PAIR;
  CUtensorMap ta, tb;
  if (!tmap_2d(&ta, x_g, H, R, BK, BM) || !tmap_3d(&tb, w13, H, 2 * I, E, BK, 128)) return cudaErrorInvalidValue;
  GemmArgs g = base_args(E, offsets, tile_off, status);
  g.N = I;
  g.K = H;
  g.I = I;
  g.out0 = hu;
  g.ld0 = 2LL * I;
  g.out1 = act_hi;
  g.out2 = act_lo;
  g.ld1 = I;
  // TMA store maps of the outputs: h | u fp32 [R][2I] (SW128), a hi / lo bf16 [R][I] (SW64)
  CUtensorMap thu, tah, tal;
  if (!tmap_out(&thu, hu, 2ULL * I, R, true) || !tmap_out(&tah, act_hi, I, R, false) ||
      !tmap_out(&tal, act_lo, I, R, false))
    return cudaErrorInvalidValue;
  if (pair)
    return launch_pair<EPI_SWIGLU, SPLIT_NONE>(ta, ta, tb, thu, tah, tal, g, pair_tiles_bound(R, E) * (I / 128), n_sm,
                                               st);
  const int bound = row_tiles_bound(R, E) * (I / 128);
  return launch<MODE_ROWS, EPI_SWIGLU, SPLIT_NONE, 256>(ta, ta, tb, tb, g, std::min(bound, n_sm), st, &thu, &tah,
                                                        &tal);
}

cudaError_t launch_gemm2(const void* act_hi, const void* act_lo, const void* w2, int R, int H, int I, int E,
                         const int32_t* offsets, const int32_t* tile_off, float* out, int* status, int n_sm,
                         int variant, bool f16, cudaStream_t st) {
  const bool pair = variant == GEMM_ROWS_PAIR;
  if (f16 && variant != GEMM_NARROW) return cudaErrorInvalidValue;
  if (variant == GEMM_NARROW) {
    // W2 [E][H][I] K-major, 128-row boxes (one CTA's half of a 256-row weight tile)
    CUtensorMap tw;
    if (!tmap_3d(&tw, w2, I, H, E, BK, 128)) return cudaErrorInvalidValue;
    GemmArgs g = base_args(E, offsets, tile_off, status);
    g.N = H;
    g.K = I;
    g.out0 = out;
    g.ld0 = H;
    g.ticket = work_counter(status, CNT_GEMM2);
    if (f16) {
      // fp16 a (one value, 11 significant bits) against an fp16 copy of W2: one MMA per K step
      // (the TMA copies are bitwise: the bf16 maps serve any 16-bit element)
      g.f16 = 1;
      if (narrow_short_rows(R, E))
        return launch_narrow<false, false, 256, EPI_F32_PAIRED>(tw, act_hi, nullptr, I, g, R, n_sm, st);
      return launch_narrow<false, false, 256>(tw, act_hi, nullptr, I, g, R, n_sm, st);
    }
    if (narrow_deep(R, E))
      return launch_narrow<false, true, 192, EPI_F32_PAIRED>(tw, act_hi, act_lo, I, g, R, n_sm, st);
    if (narrow_short_rows(R, E))
      return launch_narrow<false, true, 256, EPI_F32_PAIRED>(tw, act_hi, act_lo, I, g, R, n_sm, st);
    return launch_narrow<false, true, 256>(tw, act_hi, act_lo, I, g, R, n_sm, st);
  }
  CUtensorMap ta, ta2, tb;
  if (!tmap_2d(&ta, act_hi, I, R, BK, BM) || !tmap_2d(&ta2, act_lo, I, R, BK, BM) ||
      !tmap_3d(&tb, w2, I, H, E, BK, pair ? 128 : 256))
    return cudaErrorInvalidValue;
  GemmArgs g = base_args(E, offsets, tile_off, status);
  g.N = H;
  g.K = I;
  g.out0 = out;
  g.ld0 = H;
  CUtensorMap to;
  if (!tmap_out(&to, out, H, R, true)) return cudaErrorInvalidValue;
  if (pair)
    return launch_pair<EPI_F32, SPLIT_A>(ta, ta2, tb, to, to, to, g, pair_tiles_bound(R, E) * ((H + 255) / 256), n_sm,
                                         st);
  const int bound = row_tiles_bound(R, E) * ((H + 255) / 256);
  return launch<MODE_ROWS, EPI_F32, SPLIT_A, 256>(ta, ta2, tb, tb, g, std::min(bound, n_sm), st, &to);
}

cudaError_t launch_dgrad_swiglu(const void* dy_g, const void* w2, int R, int H, int I, int E,
                                const int32_t* offsets, const int32_t* tile_off, const float* hu,
                                const float* gate_row, void* dhu_hi, void* dhu_lo, void* gact_hi, void* gact_lo,
                                float* dg_part, int* status, int n_sm, cudaStream_t st) {
  CUtensorMap ta, tb;
  // A = dY_g [R][H] (K = H, K-major); B = W2[e] [H][I] seen as [K][N] (N contiguous)
  if (!tmap_2d(&ta, dy_g, H, R, BK, BM) || !tmap_3d(&tb, w2, I, H, E, 64, BK)) return cudaErrorInvalidValue;
  GemmArgs g = base_args(E, offsets, tile_off, status);
  g.N = I;
  g.K = H;
  g.I = I;
  g.out0 = dhu_hi;
  g.out1 = dhu_lo;
  g.ld0 = 2LL * I;
  g.out2 = gact_hi;
  g.out3 = gact_lo;
  g.ld1 = I;
  g.out4 = dg_part;
  g.ld2 = (I + 255) / 256;  // one partial per 256-column tile (the last may hold 128)
  g.hu = hu;
  g.gate_row = gate_row;
  const int bound = row_tiles_bound(R, E) * ((I + 255) / 256);
  return launch<MODE_DGRAD, EPI_SWIGLU_BWD, SPLIT_NONE, 256>(ta, ta, tb, tb, g, std::min(bound, n_sm), st);
}

cudaError_t launch_dgrad_x(const void* dhu_hi, const void* dhu_lo, const void* w13, int R, int H, int I, int E,
                           const int32_t* offsets, const int32_t* tile_off, float* dx_g, int* status, int n_sm,
                           int variant, cudaStream_t st) {
  if (variant == GEMM_NARROW) {
    // W13[e] [2I][H] as an MN-major W (64 x 64 boxes)
    CUtensorMap tw;
    if (!tmap_3d(&tw, w13, H, 2 * I, E, 64, BK)) return cudaErrorInvalidValue;
    GemmArgs g = base_args(E, offsets, tile_off, status);
    g.N = H;
    g.K = 2 * I;
    g.out0 = dx_g;
    g.ld0 = H;
    g.ticket = work_counter(status, CNT_DGRAD_X);
    if (dhu_lo == nullptr) return launch_narrow<true, false, 256>(tw, dhu_hi, nullptr, 2 * I, g, R, n_sm, st);
    if (narrow_deep(R, E))
      return launch_narrow<true, true, 192, EPI_F32_PAIRED>(tw, dhu_hi, dhu_lo, 2 * I, g, R, n_sm, st);
    if (narrow_short_rows(R, E))
      return launch_narrow<true, true, 256, EPI_F32_PAIRED>(tw, dhu_hi, dhu_lo, 2 * I, g, R, n_sm, st);
    return launch_narrow<true, true, 256>(tw, dhu_hi, dhu_lo, 2 * I, g, R, n_sm, st);
  }
  CUtensorMap ta, ta2, tb;
  // A = dHU [R][2I] (K = 2I) as hi + lo (or a single bf16 tensor when dhu_lo is null);
  // B = W13[e] [2I][H] seen as [K][N] (N = H contiguous)
  if (!tmap_2d(&ta, dhu_hi, 2 * I, R, BK, BM) || !tmap_3d(&tb, w13, H, 2 * I, E, 64, BK)) return cudaErrorInvalidValue;
  ta2 = ta;
  if (dhu_lo != nullptr && !tmap_2d(&ta2, dhu_lo, 2 * I, R, BK, BM)) return cudaErrorInvalidValue;
  GemmArgs g = base_args(E, offsets, tile_off, status);
  g.N = H;
  g.K = 2 * I;
  g.out0 = dx_g;
  g.ld0 = H;
  const int bound = row_tiles_bound(R, E) * ((H + 255) / 256);
  CUtensorMap to;
  if (!tmap_out(&to, dx_g, H, R, true)) return cudaErrorInvalidValue;
  if (dhu_lo == nullptr)
    return launch<MODE_DGRAD, EPI_F32, SPLIT_NONE, 256>(ta, ta, tb, tb, g, std::min(bound, n_sm), st, &to);
  return launch<MODE_DGRAD, EPI_F32, SPLIT_A, 256>(ta, ta2, tb, tb, g, std::min(bound, n_sm), st, &to);
}

cudaError_t launch_wgrad(const void* a_hi, const void* a_lo, int M, const void* b_hi, const void* b_lo, int N, int R,
                         int E, const int32_t* offsets, void* dw, int out_f32, int* status, int* strip_counter,
                         bool pair, int n_sm, cudaStream_t st) {
  constexpr int WBN = 128;
  CUtensorMap ta, ta2, tb, tb2;
  if (!tmap_2d(&ta, a_hi, M, R, 64, BK) || !tmap_2d(&tb, b_hi, N, R, 64, BK)) return cudaErrorInvalidValue;
  ta2 = ta;
  tb2 = tb;
  if (a_lo && !tmap_2d(&ta2, a_lo, M, R, 64, BK)) return cudaErrorInvalidValue;
  if (b_lo && !tmap_2d(&tb2, b_lo, N, R, 64, BK)) return cudaErrorInvalidValue;
  // at most one operand is a hi/lo pair: it is the stationary one (A when neither is)
  if (a_lo != nullptr && b_lo != nullptr) return cudaErrorInvalidValue;
  const bool split = a_lo != nullptr || b_lo != nullptr;
  const bool stat_a = a_lo != nullptr || !split;
  (void)WBN;
  WgradArgs g;
  g.M = M;
  g.N = N;
  g.E = E;
  g.offsets = offsets;
  g.out = dw;
  g.status = status;
  g.strip_counter = strip_counter;
  if (strip_counter == nullptr) return cudaErrorInvalidValue;
  const size_t smem = wgrad_smem_bytes(E);
  if (pair && M % 256 == 0 && N % 256 == 0) {
    // CTA pairs: 256 x 256 output tiles, each CTA half of both operands; the output as
    // [E*N rows][M] for the epilogue's 32 x 32 TMA stores
    const int pstrips = E * (stat_a ? M / 256 : N / 256);
    if (pstrips <= 0) return cudaSuccess;
    CUtensorMap to;
    {
      const uint64_t dims[2] = {(uint64_t)M, (uint64_t)E * N};
      const uint64_t strides[1] = {(uint64_t)M * (out_f32 ? 4 : 2)};
      const uint32_t box[2] = {32, 32};
      if (!make_tmap(&to, dw, 2, dims, strides, box,
                     out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    }
    // the largest shared memory of any E: six stages up to WGP_E_SIX experts, five up to 1024
    constexpr size_t smem_max = std::max(wgrad_pair_smem_bytes(WGP_E_SIX), wgrad_pair_smem_bytes(1024));
    static_assert(smem_max <= 232448, "shared memory budget");
    auto run_pair = [&](auto kern) {
      cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
      if (err != cudaSuccess) return err;
      cudaLaunchConfig_t cfg{};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.blockDim = dim3(WGP_THREADS, 1, 1);
      cfg.dynamicSmemBytes = wgrad_pair_smem_bytes(E);
      cfg.stream = st;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      cfg.gridDim = dim3(2 * std::max(1, n_sm / 2), 1, 1);
      int clusters = 0;
      if ((err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return err;
      cfg.gridDim = dim3(2 * std::min(pstrips, std::max(1, clusters)), 1, 1);
      if ((err = cudaLaunchKernelEx(&cfg, kern, ta, ta2, tb, tb2, to, g)) != cudaSuccess) return err;
      return cudaGetLastError();
    };
    if (!split) return out_f32 ? run_pair(wgrad_pair_kernel<true, true, false>) : run_pair(wgrad_pair_kernel<true, false, false>);
    if (a_lo) return out_f32 ? run_pair(wgrad_pair_kernel<true, true>) : run_pair(wgrad_pair_kernel<true, false>);
    return out_f32 ? run_pair(wgrad_pair_kernel<false, true>) : run_pair(wgrad_pair_kernel<false, false>);
  }
  const int strips = E * (stat_a ? M / 128 : N / 128);
  const int grid = std::min(strips, n_sm);
  if (grid <= 0) return cudaSuccess;
  auto run = [&](auto kern) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wgrad_smem_bytes(1024));
    if (err != cudaSuccess) return err;
    kern<<<grid, WG_THREADS, smem, st>>>(ta, ta2, tb, tb2, g);
    return cudaGetLastError();
  };
  static_assert(wgrad_smem_bytes(1024) <= 232448, "shared memory budget");
  if (!split) return out_f32 ? run(wgrad_kernel<true, true, false>) : run(wgrad_kernel<true, false, false>);
  if (a_lo) return out_f32 ? run(wgrad_kernel<true, true>) : run(wgrad_kernel<true, false>);
  return out_f32 ? run(wgrad_kernel<false, true>) : run(wgrad_kernel<false, false>);
}

// Ring GEMM1 on the narrow-segment CTA-pair kernel: chunks of at most 256 rows of each expert's
// segment in a minibatch, 128 intermediate indices (64 gate + 64 up rows per CTA) per pair tile,
// or, where the plain forward takes the paired SwiGLU form (>= 384 rows per expert, whole
// 256-index tiles), 256 (128 gate + 128 up rows per CTA).
constexpr int RING_NARROW_NMAX = 256;

int ring_chunk_rows(int variant) { return variant == GEMM_NARROW ? RING_NARROW_NMAX : BM; }

bool ring_gemm1_paired(int variant, int R, int E, int I) {
  return variant == GEMM_NARROW && (long long)R >= 384LL * E && I % 256 == 0;
}

int ring_tiles_per_chunk(int variant, int R, int E, int I) {
  return ring_gemm1_paired(variant, R, E, I) ? I / 256 : I / 128;
}

namespace {

template <int EPI>
cudaError_t launch_ring_gemm1_narrow(const RingArgs& ra, const void* w13, float* hu, void* act_hi, void* act_lo,
                                     int* status, int n_sm, cudaStream_t st) {
  using C = NarrowCfg<false, false, RING_NARROW_NMAX, EPI>;
  static_assert(C::smem_bytes(1024) <= 232448, "shared memory budget");
  const uint64_t ring_rows = (uint64_t)ra.ring_slots * ra.mb_rows;
  CUtensorMap tw, tx, txs;
  if (!tmap_w13_gate_up(&tw, w13, ra.H, ra.I, ra.E, EPI == EPI_SWIGLU_PAIRED ? 128 : 64) ||
      !tmap_2d(&tx, ra.ring, ra.H, ring_rows, BK, NARROW_XBOX) ||
      !tmap_2d(&txs, ra.ring, ra.H, ring_rows, BK, NARROW_XBOX_S))
    return cudaErrorInvalidValue;
  // whole clusters of gathering CTAs, at least one pair of GEMM CTAs
  if (ra.comm_ctas < 2 || ra.comm_ctas % 2 != 0 || ra.comm_ctas + 2 > n_sm) return cudaErrorInvalidValue;
  GemmArgs g = base_args(ra.E, nullptr, nullptr, status);
  g.N = ra.I;
  g.K = ra.H;
  g.I = ra.I;
  g.out0 = hu;
  g.ld0 = 2LL * ra.I;
  g.out1 = act_hi;
  g.out2 = act_lo;
  g.ld1 = ra.I;
  g.comm_ctas = ra.comm_ctas;
  g.n_mb = ra.n_mb;
  g.mb_rows = ra.mb_rows;
  g.ring_slots = ra.ring_slots;
  g.ring_shift = ra.ring_shift;
  g.R = ra.R;
  g.k_top = ra.k;
  g.H = ra.H;
  g.mb_off = ra.mb_off;
  g.mb_toff = ra.mb_toff;
  g.mb_start = ra.mb_start;
  g.gathered = ra.gathered;
  g.consumed = ra.consumed;
  g.consume_per_tile = 2 * C::EPI_WARPS;  // every epilogue warp of both CTAs of the pair
  g.ticket = ra.ticket;
  g.x = reinterpret_cast<const __nv_bfloat16*>(ra.x);
  g.src_of = ra.src_of;
  g.ring = reinterpret_cast<__nv_bfloat16*>(ra.ring);
  auto kern = gemm_narrow_kernel<false, false, RING_NARROW_NMAX, EPI, NARROW_RING_GEMM1>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem_bytes(1024));
  if (err != cudaSuccess) return err;
  // gathering and GEMM CTAs wait on each other: the launch is cooperative (all CTAs resident at
  // once), in clusters of two, one CTA per SM
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::smem_bytes(ra.E);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  static int max_clusters[64] = {0};  // co-resident clusters of this kernel, per device
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_clusters[dev] == 0) {
    cfg.gridDim = dim3(2 * std::max(1, n_sm / 2), 1, 1);
    int clusters = 0;
    if ((err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return err;
    max_clusters[dev] = std::max(1, clusters);
  }
  const int pairs = max_clusters[dev] - ra.comm_ctas / 2;
  if (pairs < 1) return cudaErrorInvalidValue;
  cfg.gridDim = dim3(ra.comm_ctas + 2 * pairs, 1, 1);
  err = cudaLaunchKernelEx(&cfg, kern, tw, tx, tx, txs, txs, g);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ring_gemm1(const RingArgs& ra, const void* w13, float* hu, void* act_hi, void* act_lo,
                              int* status, int n_sm, int variant, cudaStream_t st) {
  if (ring_gemm1_paired(variant, ra.R, ra.E, ra.I))
    return launch_ring_gemm1_narrow<EPI_SWIGLU_PAIRED>(ra, w13, hu, act_hi, act_lo, status, n_sm, st);
  if (variant == GEMM_NARROW)
    return launch_ring_gemm1_narrow<EPI_SWIGLU>(ra, w13, hu, act_hi, act_lo, status, n_sm, st);
  using C = GemmCfg<MODE_RING, EPI_SWIGLU, SPLIT_NONE, 256>;
  CUtensorMap ta, tb;
  const uint64_t ring_rows = (uint64_t)ra.ring_slots * ra.mb_rows;
  if (!tmap_2d(&ta, ra.ring, ra.H, ring_rows, BK, BM) || !tmap_3d(&tb, w13, ra.H, 2 * ra.I, ra.E, BK, 128))
    return cudaErrorInvalidValue;
  if (ra.comm_ctas < 1 || ra.comm_ctas >= n_sm) return cudaErrorInvalidValue;
  GemmArgs g = base_args(ra.E, nullptr, nullptr, status);
  g.N = ra.I;
  g.K = ra.H;
  g.I = ra.I;
  g.out0 = hu;
  g.ld0 = 2LL * ra.I;
  g.out1 = act_hi;
  g.out2 = act_lo;
  g.ld1 = ra.I;
  g.comm_ctas = ra.comm_ctas;
  g.n_mb = ra.n_mb;
  g.mb_rows = ra.mb_rows;
  g.ring_slots = ra.ring_slots;
  g.ring_shift = ra.ring_shift;
  g.R = ra.R;
  g.k_top = ra.k;
  g.H = ra.H;
  g.mb_off = ra.mb_off;
  g.mb_toff = ra.mb_toff;
  g.mb_start = ra.mb_start;
  g.gathered = ra.gathered;
  g.consumed = ra.consumed;
  g.consume_per_tile = 4;  // the four epilogue warps of the CTA
  g.x = reinterpret_cast<const __nv_bfloat16*>(ra.x);
  g.src_of = ra.src_of;
  g.ring = reinterpret_cast<__nv_bfloat16*>(ra.ring);
  auto kern = gemm_kernel<MODE_RING, EPI_SWIGLU, SPLIT_NONE, 256>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem_bytes(1024));
  if (err != cudaSuccess) return err;
  // gathering and GEMM CTAs wait on each other: all of them must be resident at once
  // one pointer per kernel parameter: tmA, tmA2, tmB, tmB2, tmO, tmO1, tmO2, args
  void* params[] = {(void*)&ta, (void*)&ta, (void*)&tb, (void*)&tb, (void*)&ta, (void*)&ta, (void*)&ta, (void*)&g};
  return cudaLaunchCooperativeKernel((const void*)kern, dim3(n_sm), dim3(C::THREADS), params,
                                     C::smem_bytes(ra.E), st);
}

// ----------------------------------------------------------------------------- wait test
__global__ void test_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
    // nothing ever arrives on `bar`: the wait must give up and report
    mbar_wait(smem_u32(&bar), 0, &abort_flag, status, SITE_TEST_WAIT, limit_ns);
  }
}

cudaError_t launch_test_wait(int* status, long long limit_ns, cudaStream_t st) {
  test_wait_kernel<<<1, 32, 0, st>>>(status, (unsigned long long)limit_ns);
  return cudaGetLastError();
}

}  // namespace mok
