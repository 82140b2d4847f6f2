// Host launcher of the persistent ring forward (ring_forward_kernel, gemm_narrow.cuh): the token
// gather, GEMM1 + SwiGLU, GEMM2 and the weighted merge in one cooperative launch.
#include <algorithm>

#include "gemm_narrow.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace mok {

namespace {

template <int EPI1, int EPI2>
cudaError_t launch_ring_forward_t(const RingArgs& ra, const void* w13, const void* w2, float* hu, void* act_hi,
                                  void* act_lo, float* o, const float* gates, const int32_t* row_of, int T,
                                  void* y, int* status, int n_sm, cudaStream_t st) {
  using RC = RingFwdCfg<EPI1, EPI2>;
  using C1 = typename RC::C1;
  using C2 = typename RC::C2;
  static_assert(RC::smem_bytes(1024) <= 232448, "shared memory budget");
  const uint64_t ring_rows = (uint64_t)ra.ring_slots * ra.mb_rows;
  CUtensorMap t1w, t1x, t1xs, t2w, t2x, t2x2, t2xs, t2x2s;
  if (!tmap_w13_gate_up(&t1w, w13, ra.H, ra.I, ra.E, EPI1 == EPI_SWIGLU_PAIRED ? 128 : 64) ||
      !tmap_2d(&t1x, ra.ring, ra.H, ring_rows, BK, NARROW_XBOX) ||
      !tmap_2d(&t1xs, ra.ring, ra.H, ring_rows, BK, NARROW_XBOX_S) ||
      !tmap_3d(&t2w, w2, ra.I, ra.H, ra.E, BK, 128) ||
      !tmap_2d(&t2x, act_hi, ra.I, ra.R, BK, NARROW_XBOX) || !tmap_2d(&t2xs, act_hi, ra.I, ra.R, BK, NARROW_XBOX_S) ||
      !tmap_2d(&t2x2, act_lo, ra.I, ra.R, BK, NARROW_XBOX) || !tmap_2d(&t2x2s, act_lo, ra.I, ra.R, BK, NARROW_XBOX_S))
    return cudaErrorInvalidValue;
  // whole clusters of gathering CTAs, at least one pair of GEMM CTAs; the merge takes k <= 8
  if (ra.comm_ctas < 2 || ra.comm_ctas % 2 != 0 || ra.comm_ctas + 2 > n_sm || ra.k > 8) return cudaErrorInvalidValue;
  // GEMM1 on the ring, as the GEMM1-only ring launch
  GemmArgs a1 = base_args(ra.E, nullptr, nullptr, status);
  a1.N = ra.I;
  a1.K = ra.H;
  a1.I = ra.I;
  a1.out0 = hu;
  a1.ld0 = 2LL * ra.I;
  a1.out1 = act_hi;
  a1.out2 = act_lo;
  a1.ld1 = ra.I;
  a1.comm_ctas = ra.comm_ctas;
  a1.n_mb = ra.n_mb;
  a1.mb_rows = ra.mb_rows;
  a1.ring_slots = ra.ring_slots;
  a1.ring_shift = ra.ring_shift;
  a1.R = ra.R;
  a1.k_top = ra.k;
  a1.H = ra.H;
  a1.mb_off = ra.mb_off;
  a1.mb_toff = ra.mb_toff;
  a1.mb_start = ra.mb_start;
  a1.gathered = ra.gathered;
  a1.consumed = ra.consumed;
  a1.consume_per_tile = 2 * C1::EPI_WARPS;
  a1.ticket = ra.ticket;
  a1.fence_out = 1;  // GEMM2 reads a minibatch's rows of a once its tiles have counted out
  a1.x = reinterpret_cast<const __nv_bfloat16*>(ra.x);
  a1.src_of = ra.src_of;
  a1.ring = reinterpret_cast<__nv_bfloat16*>(ra.ring);
  // GEMM2 over the same row chunks, minibatch by minibatch
  GemmArgs a2 = base_args(ra.E, nullptr, nullptr, status);
  a2.N = ra.H;
  a2.K = ra.I;
  a2.out0 = o;
  a2.ld0 = ra.H;
  a2.n_mb = ra.n_mb;
  a2.mb_rows = ra.mb_rows;
  a2.ring_slots = ra.ring_slots;
  a2.ring_shift = ra.ring_shift;
  a2.R = ra.R;
  a2.k_top = ra.k;
  a2.H = ra.H;
  a2.mb_off = ra.mb_off;
  a2.mb_toff = ra.mb_toff;
  a2.mb_start = ra.mb_start;
  a2.consumed = ra.consumed;
  a2.consume_per_tile = 2 * C1::EPI_WARPS;
  a2.ticket = ra.ticket2;
  a2.mb_tiles1 = C1::m_tiles(a1);
  a2.done = ra.done;
  RingCombineArgs cb;
  cb.o = o;
  cb.gates = gates;
  cb.row_of = row_of;
  cb.T = T;
  cb.k = ra.k;
  cb.vec_per_row = ra.H / 8;
  cb.y = reinterpret_cast<__nv_bfloat16*>(y);

  auto kern = ring_forward_kernel<EPI1, EPI2>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RC::smem_bytes(1024));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.blockDim = dim3(RC::THREADS, 1, 1);
  cfg.dynamicSmemBytes = RC::smem_bytes(ra.E);
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
  err = cudaLaunchKernelEx(&cfg, kern, t1w, t1x, t1xs, t2w, t2x, t2x2, t2xs, t2x2s, a1, a2, cb);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ring_forward(const RingArgs& ra, const void* w13, const void* w2, float* hu, void* act_hi,
                                void* act_lo, float* o, const float* gates, const int32_t* row_of, int T, void* y,
                                int* status, int n_sm, cudaStream_t st) {
  // the forms the separate launches take: GEMM1 paired from 384 rows per expert (whole 256-index
  // tiles), GEMM2 with two weight tiles per pair tile up to 160 rows per expert
  const bool paired1 = ring_gemm1_paired(GEMM_NARROW, ra.R, ra.E, ra.I);
  const bool paired2 = narrow_short_rows(ra.R, ra.E);
  if (paired1 && !paired2)
    return launch_ring_forward_t<EPI_SWIGLU_PAIRED, EPI_F32>(ra, w13, w2, hu, act_hi, act_lo, o, gates, row_of, T, y,
                                                             status, n_sm, st);
  if (!paired1 && !paired2)
    return launch_ring_forward_t<EPI_SWIGLU, EPI_F32>(ra, w13, w2, hu, act_hi, act_lo, o, gates, row_of, T, y, status,
                                                      n_sm, st);
  if (!paired1 && paired2)
    return launch_ring_forward_t<EPI_SWIGLU, EPI_F32_PAIRED>(ra, w13, w2, hu, act_hi, act_lo, o, gates, row_of, T, y,
                                                             status, n_sm, st);
  return cudaErrorInvalidValue;  // paired GEMM1 needs >= 384 rows per expert, paired GEMM2 <= 160
}

}  // namespace mok
