// Host launchers of the block-scaled MXFP8 grouped GEMMs (gemm_mx.cuh): TMA descriptors of the
// E4M3 weights and row operands, and the kernel configurations of GEMM1 and GEMM2.
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

// Chunks of at most 192 rows: one chunk per expert at the DSV3 layer (97..162 rows per expert).
constexpr int MX_NMAX = 192;
constexpr int MX_STAGES_SWIGLU = 3;   // 58 KB stages: 32 KB of weights, 24 KB of rows, scales
constexpr int MX_STAGES_F32 = 5;      // 42 KB stages: 16 KB of weights, 24 KB of rows, scales

template <int EPI, int NMAX, int STAGES>
cudaError_t launch_mx(const CUtensorMap& tw, const CUtensorMap& tx, const MxGemmArgs& args, int n_sm,
                      cudaStream_t st) {
  using C = MxCfg<EPI, NMAX, STAGES>;
  static_assert(C::smem_bytes(1024) <= 232448, "shared memory budget");
  auto kern = gemm_mx_kernel<EPI, NMAX, STAGES>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem_bytes(1024));
  if (err != cudaSuccess) return err;
  // persistent: one CTA per SM, tiles dealt round-robin (their number is known on the device only)
  kern<<<n_sm, C::THREADS, C::smem_bytes(args.E), st>>>(tw, tx, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm1_swiglu_mxf8(const void* xq, const void* xsf, const void* w13_q, const void* w13_sf, int RP,
                                     int G, int H, int I, int E, const int32_t* offsets, const int32_t* blk_off,
                                     float* hu, void* aq, void* asf, int* status, int n_sm, cudaStream_t st) {
  CUtensorMap tw, tx;
  if (!tmap_e4m3(&tw, w13_q, H, (uint64_t)E * 2 * I, 128) || !tmap_e4m3(&tx, xq, H, RP, 32))
    return cudaErrorInvalidValue;
  MxGemmArgs a{};
  a.E = E;
  a.K = H;
  a.Nw = 2 * I;
  a.MT = I / 128;
  a.I = I;
  a.G = G;
  a.offsets = offsets;
  a.blk_off = blk_off;
  a.w_sf = static_cast<const uint8_t*>(w13_sf);
  a.x_sf = static_cast<const uint8_t*>(xsf);
  a.out = hu;
  a.ld = 2LL * I;
  a.aq = static_cast<uint8_t*>(aq);
  a.asf = static_cast<uint8_t*>(asf);
  a.status = status;
  return launch_mx<MXE_SWIGLU, MX_NMAX, MX_STAGES_SWIGLU>(tw, tx, a, n_sm, st);
}

cudaError_t launch_gemm2_mxf8(const void* aq, const void* asf, const void* w2_q, const void* w2_sf, int RP, int G,
                              int H, int I, int E, const int32_t* offsets, const int32_t* blk_off, float* o,
                              int* status, int n_sm, cudaStream_t st) {
  CUtensorMap tw, tx;
  if (!tmap_e4m3(&tw, w2_q, I, (uint64_t)E * H, 128) || !tmap_e4m3(&tx, aq, I, RP, 32)) return cudaErrorInvalidValue;
  MxGemmArgs a{};
  a.E = E;
  a.K = I;
  a.Nw = H;
  a.MT = H / 128;
  a.I = I;
  a.G = G;
  a.offsets = offsets;
  a.blk_off = blk_off;
  a.w_sf = static_cast<const uint8_t*>(w2_sf);
  a.x_sf = static_cast<const uint8_t*>(asf);
  a.out = o;
  a.ld = H;
  a.status = status;
  return launch_mx<MXE_F32, MX_NMAX, MX_STAGES_F32>(tw, tx, a, n_sm, st);
}

}  // namespace mok
