// Host-side launchers of the layer's kernels (internal to the library).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace mok {

// route.cu
cudaError_t launch_topk(const float* logits, const float* bias, const int32_t* given, int T, int E, int k,
                        int router, int renorm, float route_scale, int32_t* topk_idx, float* gates,
                        float* scores, int* status, cudaStream_t st);
cudaError_t launch_schedule(const int32_t* topk_idx, const float* gates, int R, int E, int32_t* counts,
                            int32_t* offsets, int32_t* row_of, int32_t* src_of, int32_t* tile_off,
                            float* gate_row, int* status, cudaStream_t st);
// The schedule table from ceil(R / 1024) CTAs in three launches (hist: i32 [schedule_blocks(R)][E]
// scratch); bitwise the same table as launch_schedule.
int schedule_blocks(int R);
cudaError_t launch_schedule_multi(const int32_t* topk_idx, const float* gates, int R, int E, int32_t* counts,
                                  int32_t* offsets, int32_t* row_of, int32_t* src_of, int32_t* tile_off,
                                  float* gate_row, int32_t* hist, int* status, cudaStream_t st);
cudaError_t launch_router_dlogits(const float* dg_part, int n_part, const int32_t* row_of,
                                  const int32_t* topk_idx, const float* gates, const float* scores, int T,
                                  int E, int k, int router, int renorm, float route_scale, float* dgates,
                                  float* dl, cudaStream_t st);
cudaError_t launch_mb_tables(const int32_t* offsets, int E, int R, int m, int n_mb, int n_tiles, int tile_rows, int32_t* mb_off,
                             int32_t* mb_toff, int32_t* mb_tiles, int32_t* mb_start, cudaStream_t st);
cudaError_t launch_router_wgrad(const float* dl, const void* x, const int32_t* offsets, const int32_t* src_of,
                                int T, int H, int E, int k, int sparse, float* dw, cudaStream_t st);

// rows.cu
// The backward's replay of the dispatched rows after a ring forward: x_rows[r] = x[src_of[r] / k]
// for r < R, except the rows the ring still holds (r >= head_rows) when the workspace's ring stamp
// is the forward's (ws_stamp == {ctx address, ctx_stamp[0]}); else every row is replayed.
cudaError_t launch_ring_replay(const void* x, const int32_t* src_of, int k, int R, int H, void* x_rows, int head_rows,
                               const unsigned long long* ws_stamp, const unsigned long long* ctx_stamp,
                               unsigned long long ctx_addr, cudaStream_t st);
// Marks the ring rows as the work of this forward: ctx_stamp[0] += 1, ws_stamp = {ctx address, ctx_stamp[0]}.
cudaError_t launch_ring_stamp(unsigned long long* ctx_stamp, unsigned long long* ws_stamp, unsigned long long ctx_addr,
                              cudaStream_t st);
cudaError_t launch_gather_rows(const void* src, const int32_t* src_of, int k, int R, int H, void* dst, int n_sm,
                               cudaStream_t st);
// out[t] = sum_j w[t][j] * rows[row_of[t*k+j]] (+ router term), rows fp32, out bf16
cudaError_t launch_combine(const float* rows, const float* w, const int32_t* row_of, int T, int k, int H,
                           const float* dl, const void* w_router, const int32_t* topk_idx, int E,
                           int dense_router, void* out, int n_sm, cudaStream_t st);

// gemm.cu
cudaError_t launch_router_gemm(const void* x, const void* w_router, int T, int H, int E, float* logits,
                               int* status, int n_sm, cudaStream_t st);
// `pair`: run the GEMM on CTA pairs (tcgen05 cta_group::2, 256-row tiles) instead of single CTAs
// (128-row tiles); same results bit for bit.
// Expert GEMM kernels (GEMM1, GEMM2, dX_g): 128-row tiles of an expert's rows on single CTAs,
// 256-row tiles on CTA pairs (GEMM1 / GEMM2), or the narrow-segment pair kernel (the expert's
// rows as the MMA's N).
enum GemmVariant { GEMM_ROWS_SINGLE = 0, GEMM_ROWS_PAIR = 1, GEMM_NARROW = 2 };
cudaError_t launch_gemm1_swiglu(const void* x_g, const void* w13, int R, int H, int I, int E,
                                const int32_t* offsets, const int32_t* tile_off, float* hu, void* act_hi,
                                void* act_lo, int* status, int n_sm, int variant, bool a_f16, cudaStream_t st);
cudaError_t launch_gemm2(const void* act_hi, const void* act_lo, const void* w2, int R, int H, int I, int E,
                         const int32_t* offsets, const int32_t* tile_off, float* out, int* status, int n_sm,
                         int variant, bool f16, cudaStream_t st);
cudaError_t launch_dgrad_swiglu(const void* dy_g, const void* w2, int R, int H, int I, int E,
                                const int32_t* offsets, const int32_t* tile_off, const float* hu,
                                const float* gate_row, void* dhu_hi, void* dhu_lo, void* gact_hi, void* gact_lo,
                                float* dg_part, int* status, int n_sm, cudaStream_t st);
cudaError_t launch_dgrad_x(const void* dhu_hi, const void* dhu_lo, const void* w13, int R, int H, int I, int E,
                           const int32_t* offsets, const int32_t* tile_off, float* dx_g, int* status, int n_sm,
                           int variant, cudaStream_t st);
// dW[e] stored transposed as out[e][n][m] (m = the output's contiguous dimension):
// out[e][n][m] = sum over rows r of expert e of A[r][m] * B[r][n]; A or B may be a hi/lo pair.
// strip_counter: a device int that is zero when the kernel starts (the single-CTA kernel deals its
// strips from it).  pair: 256 x 256 tiles on CTA pairs (M and N multiples of 256).
cudaError_t launch_wgrad(const void* a_hi, const void* a_lo, int M, const void* b_hi, const void* b_lo, int N, int R,
                         int E, const int32_t* offsets, void* dw, int out_f32, int* status, int* strip_counter,
                         bool pair, int n_sm, cudaStream_t st);
// Status region of the workspace (256 bytes, cleared at the start of every entry point): the
// status word (code, site) in ints 0..1, the work counters of dynamically dealt launches from
// int STATUS_COUNTERS on.
constexpr int STATUS_BYTES = 256;
constexpr int STATUS_COUNTERS = 16;
enum WorkCounter { CNT_WGRAD_W2 = 0, CNT_WGRAD_W13 = 1, CNT_GEMM1 = 2, CNT_GEMM2 = 3, CNT_DGRAD_X = 4 };
// The narrow-segment GEMMs (variant GEMM_NARROW of GEMM1, GEMM2 and dX_g) take their tiles from the
// work counter of their kind in the status region that `status` points to.
inline int* work_counter(int* status, WorkCounter c) { return status + STATUS_COUNTERS + (int)c; }
// Ring forward GEMM1: comm_ctas CTAs gather minibatches into the ring, the rest run GEMM1
// (SwiGLU epilogue, rows written at their global position).  Cooperative launch, grid = n_sm.
struct RingArgs {
  const void* x;
  const int32_t* src_of;
  int k, R, H, I, E;
  int mb_rows, n_mb, ring_slots, comm_ctas;
  int ring_shift;  // minibatch mb lives in slot (mb + ring_shift) % ring_slots
  void* ring;
  const int32_t* mb_off;
  const int32_t* mb_toff;
  const int32_t* mb_start;
  int32_t* gathered;
  int32_t* consumed;
  int32_t* ticket;  // the narrow ring GEMM1's tile counter (zero at launch)
  int32_t* ticket2;  // the persistent ring forward's GEMM2 tile counter (zero at launch)
  int32_t* done;     // its GEMM2 epilogue warps finished (zero at launch)
};
// variant GEMM_NARROW: the narrow-segment CTA-pair kernel (minibatch tables in chunks of
// ring_chunk_rows() rows); else the row-tile kernel (128-row tiles)
int ring_chunk_rows(int variant);
// weight tiles per row chunk of the ring GEMM1 (its form follows the plain GEMM1's: paired SwiGLU
// tiles of 256 intermediate indices from 384 rows per expert, else 128)
int ring_tiles_per_chunk(int variant, int R, int E, int I);
// the ring GEMM1 takes the paired SwiGLU form (as the plain GEMM1: >= 384 rows per expert, I a
// multiple of 256)
bool ring_gemm1_paired(int variant, int R, int E, int I);
// The narrow split-operand GEMMs (GEMM2, dX_g) take two weight tiles per pair tile when the
// experts average at most 160 rows.
inline bool narrow_short_rows(int R, int E) { return (long long)R <= 160LL * E; }
// Of those, the paired GEMM2 / dX_g take the deep form (192-row chunks, four stages) when the
// 16-bit chunk prefixes and the shared-memory budget allow it: at most 256 experts.
inline bool narrow_deep(int R, int E) {
  return narrow_short_rows(R, E) && E <= 256 && (long long)R / 192 + E < 65535;
}
// The persistent ring forward (narrow kernels, k <= 8): after the schedule and the minibatch
// tables, one cooperative launch gathers the minibatches into the ring and runs GEMM1 + SwiGLU,
// GEMM2 and the weighted merge (hu, act hi / lo, o and y as the separate launches write them).
cudaError_t launch_ring_forward(const RingArgs& ra, const void* w13, const void* w2, float* hu, void* act_hi,
                                void* act_lo, float* o, const float* gates, const int32_t* row_of, int T, void* y,
                                int* status, int n_sm, cudaStream_t st);
cudaError_t launch_ring_gemm1(const RingArgs& ra, const void* w13, float* hu, void* act_hi, void* act_lo,
                              int* status, int n_sm, int variant, cudaStream_t st);
// MXFP8 weights (mx.cu)
// w [E][N][K] bf16 -> q [E][N][K] E4M3 and 512-byte scale blocks; gate_up_I > 0 (W13, N = 2I):
// the blocks of 128 rows pair 64 gate rows with the 64 up rows of the same intermediate indices.
cudaError_t launch_quantize_weights(const void* w, void* q, void* s, int E, int N, int K, int gate_up_I, int n_sm,
                                    cudaStream_t st);
// MXFP8 backward operands (mx.cu).  src of launch_mx_quant_rows: 0 plain rows (in0, fixed
// segments of seg_len rows), 1 hi + lo rows, 2 a = silu(h) u from h | u, 3 token rows gathered by
// src_of, 4 gate_row * gathered token rows; segments from offsets / blk_off unless seg_len > 0.
cudaError_t launch_mx_block_offsets(const int32_t* offsets, int E, int32_t* blk_off, cudaStream_t st);
cudaError_t launch_mx_quant_rows(int src, int rows_bound, int C, int E, int seg_len, const int32_t* offsets,
                                 const int32_t* blk_off, const void* in0, const void* in1, const float* hu,
                                 const float* gate_row, const int32_t* src_of, int k, void* out, int n_sm,
                                 cudaStream_t st);
cudaError_t launch_mx_quant_cols(const void* hi, const void* lo, long long R, int C, void* out, int n_sm,
                                 cudaStream_t st);
cudaError_t launch_gather_rows_mx(const void* src, const int32_t* src_of, int k, int R, int H, void* dst, int n_sm,
                                  cudaStream_t st);
// MXFP8 forward on the FP8 tensor path (mx.cu, gemm_mx.cu): E4M3 row operands in the padded row
// space of mx_tiles.h (blk_off from launch_mx_block_offsets), scale blocks of RP / 32 + 4 row groups.
cudaError_t launch_gather_rows_mxf8(const void* x, const int32_t* src_of, const int32_t* topk_idx,
                                    const int32_t* offsets, const int32_t* blk_off, int k, int R, int H, int E,
                                    void* xq, void* xsf, cudaStream_t st);
cudaError_t launch_gemm1_swiglu_mxf8(const void* xq, const void* xsf, const void* w13_q, const void* w13_sf, int RP,
                                     int G, int R, int H, int I, int E, const int32_t* offsets, const int32_t* blk_off,
                                     float* hu, void* aq, void* asf, int* status, int n_sm, cudaStream_t st);
cudaError_t launch_gemm2_mxf8(const void* aq, const void* asf, const void* w2_q, const void* w2_sf, int RP, int G,
                              int R, int H, int I, int E, const int32_t* offsets, const int32_t* blk_off, float* o,
                              int* status, int n_sm, cudaStream_t st);
// MXFP8 backward on the FP8 tensor path: dA' = dY_g W2[e] with the SwiGLU backward (dh | du as bf16
// hi / lo and as E4M3 along 2I, partial gate gradients per 128 intermediate indices), and
// dX_g = dHU W13[e]; the weights transposed and quantised along their reduction (launch_quantize_transpose).
cudaError_t launch_dgrad_swiglu_mxf8(const void* dyq, const void* dysf, const void* w2t_q, const void* w2t_sf, int RP,
                                     int G, int R, int H, int I, int E, const int32_t* offsets, const int32_t* blk_off,
                                     const float* hu, const float* gate_row, void* dhu_hi, void* dhu_lo, void* dhuq,
                                     void* dhusf, float* dg_part, int* status, int n_sm, cudaStream_t st);
cudaError_t launch_dgrad_x_mxf8(const void* dhuq, const void* dhusf, const void* w13t_q, const void* w13t_sf, int RP,
                                int G, int R, int H, int I, int E, const int32_t* offsets, const int32_t* blk_off,
                                float* dx_g, int* status, int n_sm, cudaStream_t st);
// w [E][N][K] bf16 -> wt [E][K][N] E4M3 quantised in 32-blocks along N, scales [E][K/128][N/128][512].
cudaError_t launch_quantize_transpose(const void* w, void* wt_q, void* wt_s, int E, int N, int K, int n_sm,
                                      cudaStream_t st);
// src [n] bf16 -> dst [n] fp16 (round to nearest even; exact for bf16 values of magnitude 2^-14 .. 65504)
cudaError_t launch_bf16_to_f16(const void* src, void* dst, long long n, int n_sm, cudaStream_t st);
cudaError_t launch_test_wait(int* status, long long limit_ns, cudaStream_t st);

}  // namespace mok
