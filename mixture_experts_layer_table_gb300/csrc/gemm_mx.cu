// Host launchers of the block-scaled MXFP8 grouped GEMMs (gemm_mx.cuh): TMA descriptors of the E4M3
// weights, the padded row operands and their scale blocks, and the kernel configurations of GEMM1,
// GEMM2 and the two data-gradient GEMMs of the backward.
#include <cuda.h>

#include <algorithm>

#include "gemm_mx.cuh"
#include "kernels.cuh"
#include "tmap.cuh"

namespace mok {

namespace {

// E4M3 bytes [rows][cols] with 128-byte swizzle, boxes of 128 bytes x box_rows rows.
bool tmap_e4m3(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {cols};
  const uint32_t box[2] = {MX_BK, box_rows};
  return make_tmap(m, base, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_128B);
}

// W13 E4M3 [E][2I][H] seen as [E][2][I][H]: one box = 64 gate rows and their 64 up rows.
bool tmap_e4m3_gate_up(CUtensorMap* m, const void* w13_q, uint64_t H, uint64_t I, uint64_t E) {
  const uint64_t dims[4] = {H, I, 2, E};
  const uint64_t strides[3] = {H, I * H, 2 * I * H};
  const uint32_t box[4] = {MX_BK, 64, 2, 1};
  return make_tmap(m, w13_q, 4, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_128B);
}

// `blocks` 512-byte scale blocks seen as [blocks][4][128] bytes, one block per box, no swizzle.
bool tmap_sf_blocks(CUtensorMap* m, const void* base, uint64_t blocks) {
  const uint64_t dims[3] = {128, 4, blocks};
  const uint64_t strides[2] = {128, MX_SF_BLOCK};
  const uint32_t box[3] = {128, 4, 1};
  return make_tmap(m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Chunks of at most 192 rows (one per expert at the DSV3 layer, 97..162 rows per expert); stage
// rings as deep as shared memory allows (30 KB stages: 16 KB of weights, up to 96 rows, scales).
constexpr int MX_NMAX = 192;
constexpr int MX_STAGES_SWIGLU = 6;
constexpr int MX_STAGES_BWD = 6;
constexpr int MX_STAGES = 7;

MxGemmArgs mx_args(int E, int K, int MT, int Nw, int I, int sfa_tiles, const int32_t* offsets, const int32_t* blk_off,
                   int* status) {
  MxGemmArgs a{};
  a.E = E;
  a.K = K;
  a.MT = MT;
  a.Nw = Nw;
  a.I = I;
  a.sfa_tiles = sfa_tiles;
  a.offsets = offsets;
  a.blk_off = blk_off;
  a.status = status;
  return a;
}

template <int EPI, int NMAX, int STAGES>
cudaError_t launch_mx(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& tws, const CUtensorMap& txs,
                      const MxGemmArgs& args, int R, int n_sm, cudaStream_t st) {
  using C = MxCfg<EPI, NMAX, STAGES>;
  static_assert(C::smem_bytes(1024) <= 232448, "shared memory budget");
  const int bound = ((R + NMAX - 1) / NMAX + args.E) * args.MT;  // pair tiles at most
  if (R <= 0 || bound <= 0) return cudaSuccess;
  auto kern = gemm_mx_kernel<EPI, NMAX, STAGES>;
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
  static int max_pairs[64] = {0};  // co-resident pairs of this kernel, per device
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_pairs[dev] == 0) {
    cfg.gridDim = dim3(2 * std::max(1, n_sm / 2), 1, 1);
    int clusters = 0;
    if ((err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return err;
    max_pairs[dev] = std::max(1, clusters);
  }
  cfg.gridDim = dim3(2 * std::min(bound, max_pairs[dev]), 1, 1);
  err = cudaLaunchKernelEx(&cfg, kern, tw, tx, tws, txs, args);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm1_swiglu_mxf8(const void* xq, const void* xsf, const void* w13_q, const void* w13_sf, int RP,
                                     int G, int R, int H, int I, int E, const int32_t* offsets, const int32_t* blk_off,
                                     float* hu, void* aq, void* asf, int* status, int n_sm, cudaStream_t st) {
  CUtensorMap tw, tx, tws, txs;
  if (!tmap_e4m3_gate_up(&tw, w13_q, H, I, E) || !tmap_e4m3(&tx, xq, H, RP, 32) ||
      !tmap_sf_blocks(&tws, w13_sf, (uint64_t)E * (I / 64) * (H / MX_BK)) ||
      !tmap_sf_blocks(&txs, xsf, (uint64_t)G * (H / MX_BK)))
    return cudaErrorInvalidValue;
  MxGemmArgs a = mx_args(E, H, I / 128, 2 * I, I, I / 64, offsets, blk_off, status);
  a.out = hu;
  a.ld = 2LL * I;
  a.q = static_cast<uint8_t*>(aq);
  a.qsf = static_cast<uint8_t*>(asf);
  return launch_mx<MXE_SWIGLU, MX_NMAX, MX_STAGES_SWIGLU>(tw, tx, tws, txs, a, R, n_sm, st);
}

cudaError_t launch_gemm2_mxf8(const void* aq, const void* asf, const void* w2_q, const void* w2_sf, int RP, int G,
                              int R, int H, int I, int E, const int32_t* offsets, const int32_t* blk_off, float* o,
                              int* status, int n_sm, cudaStream_t st) {
  CUtensorMap tw, tx, tws, txs;
  if (!tmap_e4m3(&tw, w2_q, I, (uint64_t)E * H, 128) || !tmap_e4m3(&tx, aq, I, RP, 32) ||
      !tmap_sf_blocks(&tws, w2_sf, (uint64_t)E * (H / 128) * (I / MX_BK)) ||
      !tmap_sf_blocks(&txs, asf, (uint64_t)G * (I / MX_BK)))
    return cudaErrorInvalidValue;
  MxGemmArgs a = mx_args(E, I, (H + 255) / 256, H, I, H / 128, offsets, blk_off, status);
  a.N_out = H;
  a.out = o;
  a.ld = H;
  return launch_mx<MXE_F32, MX_NMAX, MX_STAGES>(tw, tx, tws, txs, a, R, n_sm, st);
}

cudaError_t launch_dgrad_swiglu_mxf8(const void* dyq, const void* dysf, const void* w2t_q, const void* w2t_sf, int RP,
                                     int G, int R, int H, int I, int E, const int32_t* offsets, const int32_t* blk_off,
                                     const float* hu, const float* gate_row, void* dhu_hi, void* dhu_lo, void* dhuq,
                                     void* dhusf, float* dg_part, int* status, int n_sm, cudaStream_t st) {
  CUtensorMap tw, tx, tws, txs;
  if (!tmap_e4m3(&tw, w2t_q, H, (uint64_t)E * I, 128) || !tmap_e4m3(&tx, dyq, H, RP, 32) ||
      !tmap_sf_blocks(&tws, w2t_sf, (uint64_t)E * (I / 128) * (H / MX_BK)) ||
      !tmap_sf_blocks(&txs, dysf, (uint64_t)G * (H / MX_BK)))
    return cudaErrorInvalidValue;
  MxGemmArgs a = mx_args(E, H, (I + 255) / 256, I, I, I / 128, offsets, blk_off, status);
  a.hu = hu;
  a.gate_row = gate_row;
  a.dhu_hi = static_cast<__nv_bfloat16*>(dhu_hi);
  a.dhu_lo = static_cast<__nv_bfloat16*>(dhu_lo);
  a.q = static_cast<uint8_t*>(dhuq);
  a.qsf = static_cast<uint8_t*>(dhusf);
  a.dg_part = dg_part;
  return launch_mx<MXE_SWIGLU_BWD, MX_NMAX, MX_STAGES_BWD>(tw, tx, tws, txs, a, R, n_sm, st);
}

cudaError_t launch_dgrad_x_mxf8(const void* dhuq, const void* dhusf, const void* w13t_q, const void* w13t_sf, int RP,
                                int G, int R, int H, int I, int E, const int32_t* offsets, const int32_t* blk_off,
                                float* dx_g, int* status, int n_sm, cudaStream_t st) {
  CUtensorMap tw, tx, tws, txs;
  if (!tmap_e4m3(&tw, w13t_q, 2 * I, (uint64_t)E * H, 128) || !tmap_e4m3(&tx, dhuq, 2 * I, RP, 32) ||
      !tmap_sf_blocks(&tws, w13t_sf, (uint64_t)E * (H / 128) * (2 * I / MX_BK)) ||
      !tmap_sf_blocks(&txs, dhusf, (uint64_t)G * (2 * I / MX_BK)))
    return cudaErrorInvalidValue;
  MxGemmArgs a = mx_args(E, 2 * I, (H + 255) / 256, H, I, H / 128, offsets, blk_off, status);
  a.N_out = H;
  a.out = dx_g;
  a.ld = H;
  return launch_mx<MXE_F32, MX_NMAX, MX_STAGES>(tw, tx, tws, txs, a, R, n_sm, st);
}

}  // namespace mok
