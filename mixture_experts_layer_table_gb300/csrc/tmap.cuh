// TMA tensor-map encoding.  The driver's cuTensorMapEncodeTiled is found at run time through the
// runtime's entry-point query, so the library does not link libcuda.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace mok {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A tensor of `dtype` (bf16 unless given), innermost dimension first; strides in bytes for dims
// 1..rank-1; 128B swizzle unless given; out-of-bounds elements read as zero.
inline bool make_tmap(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                      const uint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  if (rank < 1 || rank > 4) return false;
  cuuint64_t d[4], s[3];
  cuuint32_t b[4], es[4] = {1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides_bytes[i];
  return enc(m, dtype, rank, const_cast<void*>(base), d, s, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Store map of a row-major output [rows][cols]: 32 x 32 boxes, fp32 with 128B swizzle (128-byte
// box rows) or bf16 with 64B swizzle (64-byte box rows), as the epilogue stages them.
inline bool tmap_out(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows, bool f32) {
  const uint64_t es = f32 ? 4 : 2;
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {cols * es};
  const uint32_t box[2] = {32, 32};
  return make_tmap(m, base, 2, dims, strides, box,
                   f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

inline bool tmap_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
             uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {inner * 2};
  const uint32_t box[2] = {box_inner, box_outer};
  return make_tmap(m, base, 2, dims, strides, box);
}

inline bool tmap_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const uint32_t box[3] = {b0, b1, 1};
  return make_tmap(m, base, 3, dims, strides, box);
}

// W13 [E][2I][H] seen as [E][2][I][H]: one box of 64 K x 64 rows x both halves brings 64 gate
// rows followed by the 64 up rows of the same intermediate indices.
inline bool tmap_w13_gate_up(CUtensorMap* m, const void* w13, uint64_t H, uint64_t I, uint64_t E, uint32_t rows = 64) {
  const uint64_t dims[4] = {H, I, 2, E};
  const uint64_t strides[3] = {H * 2, I * H * 2, 2 * I * H * 2};
  const uint32_t box[4] = {64, rows, 2, 1};
  return make_tmap(m, w13, 4, dims, strides, box);
}

}  // namespace mok
