/*
 * mok.h — C ABI of a single-GPU, deterministic mixture-of-experts layer for GB300 (sm_103a).
 *
 * One call of the layer routes T tokens of width H to k of E experts, runs each expert
 * (a SwiGLU FFN of intermediate width I) on its tokens, and merges the k expert outputs
 * of each token with the router's gate weights.  The steps and their order follow the
 * pages on Mixture-of-Kittens (MoK):
 *   - "把 MoE 通信延迟从 103μs 压到 18μs：Cursor 开源 GPU 内核 MoK" (aientropygate.com),
 *     §02: router decision -> dispatch -> grouped GEMM -> combine; the schedule step
 *     counts each expert's tokens, places them and keeps an expert's tokens together;
 *     §03 ①: the dispatch is a pull (the expert side reads the rows it needs);
 *     §03 ③: MXFP8 activation quantisation sits on the dispatch / GEMM / SwiGLU path;
 *     §04: the measured layer ends in a weighted merge.
 *   - "Mixture-of-Kittens (MoK)" (sd114.wiki), pull-dispatch section: one schedule table
 *     serves all four transfers; benchmark section: BF16 and MXFP8, router-weight
 *     gradient computed inside the SwiGLU backward; introduction: fully deterministic.
 *   - "Cursor Open-Sources Mixture-of-Kittens (MoK) ..." (aitrending.vip),
 *     "Technical Details": the same, plus the ring token buffer.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the current device; the caller owns and
 *     allocates all memory (inputs, outputs, ctx, ws).  The library never allocates,
 *     frees or synchronises inside the compute calls; everything is enqueued on `stream`
 *     (a cudaStream_t passed as void*; NULL = legacy default stream).
 *   - Row-major layouts, bf16 = IEEE bfloat16 bit patterns (uint16), f32 = IEEE float.
 *   - Return values report host-side validation only (shapes, alignment, sizes) plus
 *     launch errors.  Errors found on the device (a bounded wait that ran out, an expert
 *     index out of range) go to a status word inside `ws`; read it with mok_read_status.
 *   - Outputs are overwritten, never accumulated.  Results are bitwise reproducible for
 *     the same inputs, descriptor and device: every reduction runs in a fixed order and
 *     no floating-point atomics are used.
 *   - One call at a time per `ws`: calls that may overlap on the GPU (different streams)
 *     need a `ws` each.  Besides the temporaries, `ws` holds the status word and the work
 *     counters from which the expert GEMMs and weight-gradient kernels take their tiles
 *     (cleared by each call); two overlapping calls on one `ws` would share them and skip
 *     tiles.
 *   - No C++ exception crosses this boundary.  No global mutable state besides per-device
 *     caches of the SM count and of how many CTA pairs of each pair kernel fit at once, the
 *     driver entry point used to encode TMA descriptors, the optional per-kernel trace
 *     (mok_trace_start / mok_trace_stop) and the fixed device scratch of
 *     mok_schedule_noalloc.  The caches are filled on first use with idempotent values.
 */
#ifndef MOK_H_
#define MOK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOK_OK = 0,
  MOK_ERR_INVALID_ARG = 1,          /* null pointer, bad shape, misaligned pointer */
  MOK_ERR_UNSUPPORTED = 2,          /* shape outside what the kernels tile (see mok_layer_desc) */
  MOK_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws/ctx smaller than mok_workspace_size reports */
  MOK_ERR_CUDA = 4,                 /* a CUDA runtime/driver call or kernel launch failed */
  MOK_ERR_TIMEOUT = 5,              /* device: a bounded wait ran out (status word only) */
  MOK_ERR_INVALID_ROUTING = 6       /* device: an expert index outside [0, E) or repeated */
} mok_status;

typedef enum { MOK_ROUTER_SOFTMAX = 0, MOK_ROUTER_SIGMOID = 1 } mok_router_kind;
typedef enum { MOK_BF16 = 0, MOK_MXFP8 = 1 } mok_precision;

/* Layer descriptor.
 *   T       tokens of this call, 1 <= T
 *   H       hidden width; multiple of 128 (MOK_ERR_UNSUPPORTED otherwise)
 *   I       expert intermediate width; multiple of 128 (MOK_ERR_UNSUPPORTED otherwise).
 *           128 is one CTA's share of a CTA pair's 256-row weight tile and the K step of
 *           the MXFP8 kernels; where H or I is an odd multiple of 128 the last pair tile
 *           reads zeros past the end and stores nothing there
 *   E       routed experts, 1 <= E <= 1024
 *   k       experts per token, 1 <= k <= min(E, 16)
 *   router  mok_router_kind: softmax over E logits, or elementwise sigmoid
 *   renorm  nonzero: the k selected gates are divided by their sum
 *   route_scale  factor on every gate (1.0 for the workloads here)
 *   precision    mok_precision of the expert GEMMs
 *   ring_bytes   0: the forward gathers all T*k rows at once.  > 0: ring forward — the
 *                gathered (dispatched) rows pass through a fixed ring of this many bytes in
 *                minibatches, gathered by comm_sms CTAs while the other SMs run GEMM1 on
 *                earlier minibatches, in one persistent launch that signals through device
 *                counters ("Mixture-of-Kittens (MoK)", sd114.wiki, ring-buffer section;
 *                aientropygate.com §03 ② and ③).  The ring must hold one minibatch.
 *   minibatch    ring forward: rows per minibatch, consecutive rows of the expert-sorted
 *                order (0 = mok_min_minibatch(0, I), two full SM waves of GEMM1 tiles)
 *   flags        MOK_FLAG_WGRAD_BF16: the expert weight gradients dw13 / dw2 of
 *                mok_moe_backward are bf16 instead of the default f32.
 *                Expert GEMM kernels.  Default: GEMM1, GEMM2 and dX_g on CTA pairs with
 *                the expert's rows as the MMA's N, padded to 16 rows (tcgen05
 *                cta_group::2, 256 weight rows per pair).  MOK_FLAG_GEMM_PAIR: GEMM1 and
 *                GEMM2 on CTA pairs with 256-row tiles of an expert's rows, dX_g on
 *                single CTAs with 128-row tiles.  MOK_FLAG_GEMM_SINGLE: all three on
 *                single CTAs with 128-row tiles.  The weight gradients run on CTA pairs
 *                (256 x 256 tiles) by default and on single CTAs (128 x 128) with either
 *                flag.  Results are bitwise the same in every case.  Setting both flags
 *                is an invalid argument.
 *                MOK_FLAG_W2_F16: mok_moe_forward reads w2 as IEEE fp16 [E][H][I] (the
 *                layer's bf16 W2 converted once with mok_convert_f16, exact for weights of
 *                magnitude 2^-14 and above), keeps a = silu(h) * u as one fp16 value (11
 *                significant bits) instead of a bf16 hi / lo pair, and runs GEMM2 on fp16
 *                operands, one MMA per K step instead of two.  Default GEMM kernels and no
 *                ring only (else MOK_ERR_UNSUPPORTED); mok_moe_backward ignores the flag and
 *                takes w2 in bf16 (the backward does not read a).
 *                MOK_FLAG_RING_PERSISTENT: the ring forward (ring_bytes > 0, default GEMM
 *                kernels, k <= 8) runs GEMM2 and the weighted merge in its persistent launch
 *                too: the CTA pairs take GEMM2 tiles of each minibatch whose GEMM1 tiles have
 *                stored their rows of a, and every CTA takes tokens of the merge once every
 *                GEMM2 tile has stored its rows of o ("把 MoE 通信延迟从 103μs 压到 18μs",
 *                aientropygate.com §03 ②: one SM group for dispatch and combine, the other
 *                for the expert FFN).  Results are bitwise those of the separate launches.
 *   comm_sms     ring forward: CTAs (one per SM) that gather rows (0 = 12); even when GEMM1
 *                runs on the narrow-segment CTA-pair kernel (the default), since those
 *                CTAs are launched in clusters of two
 * T*k*max(H, 2I) must stay below 2^31 elements. */
#define MOK_FLAG_WGRAD_BF16 1
#define MOK_FLAG_GEMM_PAIR 2
#define MOK_FLAG_GEMM_SINGLE 4
#define MOK_FLAG_W2_F16 8
#define MOK_FLAG_RING_PERSISTENT 16
typedef struct {
  int32_t T, H, I, E, k;
  int32_t router;
  int32_t renorm;
  float route_scale;
  int32_t precision;
  int32_t minibatch;
  int64_t ring_bytes;
  int32_t flags;
  int32_t comm_sms;
} mok_layer_desc;

/* Byte offsets (from the base pointer) of the tensors inside ctx and ws.  ctx holds what
 * the forward saves for the backward; ws holds temporaries.  An offset of -1 means the
 * tensor is absent for this descriptor.  Every offset is a multiple of 256. */
typedef struct {
  /* ctx */
  int64_t topk_idx;   /* i32 [T][k]   selected experts, best first (ties -> lower index) */
  int64_t gates;      /* f32 [T][k]   gate weights */
  int64_t scores;     /* f32 [T][E]   router scores (softmax probabilities or sigmoids) */
  int64_t counts;     /* i32 [E]      rows per expert */
  int64_t offsets;    /* i32 [E+1]    exclusive prefix sum of counts */
  int64_t row_of;     /* i32 [T*k]    sorted row of assignment a = t*k + j */
  int64_t src_of;     /* i32 [T*k]    assignment held by sorted row r */
  int64_t tile_off;   /* i32 [E+1]    prefix sum of ceil(counts/128) (GEMM m-tiles) */
  int64_t gate_row;   /* f32 [T*k]    gate of each sorted row */
  int64_t x_g;        /* bf16 [T*k][H]  dispatched (expert-sorted) token rows */
  int64_t hu;         /* f32 [T*k][2I]  gate and up projections h | u */
  int64_t ring_stamp; /* u64 [2]      ring forward only: a count of the ring forwards on this ctx */
  int64_t ctx_bytes;
  /* ws.  "hi/lo" pairs hold v as bf16 hi = bf16(v) plus bf16 lo = bf16(v - hi), so that a
   * GEMM operand produced inside the layer keeps about 16 significant bits. */
  int64_t status;     /* i32 [64]     device status word (code, site), then per-call work counters */
  int64_t logits;     /* f32 [T][E]   router logits */
  int64_t sched;      /* i32 [ceil(T*k/1024)][E]  schedule-table scratch: per-block counts, then starts */
  int64_t act;        /* bf16 [T*k][I]  SwiGLU output a = silu(h) * u, hi part */
  int64_t act_lo;     /* bf16 [T*k][I]  lo part */
  int64_t expert_out; /* f32 [T*k][H]   expert outputs o (unweighted) */
  int64_t dy_g;       /* bf16 [T*k][H]  dispatched upstream gradient (backward) */
  int64_t dhu;        /* bf16 [T*k][2I] gradient of h | u, hi part (backward) */
  int64_t dhu_lo;     /* bf16 [T*k][2I] lo part */
  int64_t gact;       /* bf16 [T*k][I]  gate * a, operand of dW2, hi part (backward) */
  int64_t gact_lo;    /* bf16 [T*k][I]  lo part */
  int64_t dx_g;       /* f32 [T*k][H]   per-row input gradient (backward) */
  int64_t dg_part;    /* f32 [T*k][I/128] partial gate gradients per GEMM column tile (bf16: ceil(I/256) used) */
  int64_t dlogits;    /* f32 [T][E]   router logit gradient (backward) */
  /* ring forward only (-1 otherwise) */
  int64_t ring;       /* bf16 [n_mb * minibatch][H]  the dispatched rows of every minibatch: the
                          token ring is the last slots * minibatch rows, minibatch mb in slot
                          (mb + n_mb * (slots - 1)) % slots, so that the minibatches the ring still
                          holds after the forward sit at their own rows; the backward replays the
                          rest in front of them */
  int64_t mb_tables;  /* i32 [n_mb][E+1] row offsets, [n_mb][E+1] tile offsets, [n_mb] tiles,
                          [n_mb+1] tile starts (exclusive prefix of the tiles) */
  int64_t mb_counters;/* i32 [2][n_mb]  rows gathered, tile epilogues finished, per minibatch; i32
                          the GEMM1 tile counter the CTA pairs take tiles from; then (16-byte
                          aligned) u64 [2] {ctx address, ctx ring_stamp} of the forward whose rows
                          the ring holds */
  /* MXFP8 backward only (-1 otherwise): operands quantised along their GEMM's reduction
   * dimension, as exact bf16 values */
  int64_t mx_dhu_r;   /* bf16 [T*k][2I] dh | du in 32-row blocks of each expert (dW13) */
  int64_t mx_xg_r;    /* bf16 [T*k][H]  dispatched x in 32-row blocks (dW13) */
  int64_t mx_do_r;    /* bf16 [T*k][H]  gate * dY rows in 32-row blocks (dW2) */
  int64_t mx_a_r;     /* bf16 [T*k][I]  a = silu(h) * u in 32-row blocks (dW2) */
  int64_t mx_blk_off; /* i32 [E+1]      32-row blocks before each expert (forward and backward) */
  /* MXFP8 forward only (-1 otherwise): E4M3 row operands of the FP8 GEMMs in a padded row space,
   * expert e owning rows [32 mx_blk_off[e], 32 mx_blk_off[e+1]) (its rows in schedule order, then
   * zero rows); RP = 32 (ceil(T*k / 32) + E) rows, G = RP / 32 + 4 row groups.  Scales: 512-byte
   * blocks of 128 rows x 4 blocks of 32 along the row, row 32 j + l and block b at byte
   * 16 l + 4 j + b; block (g, s) holds rows 32 g .. 32 g + 127 of 128-element stage s. */
  int64_t mx_xq;      /* E4M3 [RP][H]            dispatched rows quantised along H */
  int64_t mx_xsf;     /* E8M0 [G][H/128][512]    their scale blocks */
  int64_t mx_aq;      /* E4M3 [RP][I]            a = silu(h) * u quantised along I */
  int64_t mx_asf;     /* E8M0 [G][I/128][512]    its scale blocks */
  /* MXFP8 backward, same padded row space */
  int64_t mx_dyq;     /* E4M3 [RP][H]            dispatched dY rows quantised along H */
  int64_t mx_dysf;    /* E8M0 [G][H/128][512]    their scale blocks */
  int64_t mx_dhuq;    /* E4M3 [RP][2I]           dh | du quantised along 2I */
  int64_t mx_dhusf;   /* E8M0 [G][2I/128][512]   its scale blocks */
  int64_t ws_bytes;
} mok_layout;

/* Fills *layout (and so the ctx and ws sizes) for a descriptor.  Host only. */
mok_status mok_get_layout(const mok_layer_desc* desc, mok_layout* layout);

/* The two sizes alone: *ws_bytes and *ctx_bytes are layout.ws_bytes and layout.ctx_bytes of
 * mok_get_layout.  Host only; MOK_ERR_INVALID_ARG for a null output, otherwise the descriptor's
 * validation status (outputs untouched on error). */
mok_status mok_workspace_size(const mok_layer_desc* desc, size_t* ws_bytes, size_t* ctx_bytes);

/* Router + schedule table (the "unified schedule table" of the pull-dispatch section of
 * "Mixture-of-Kittens (MoK)", sd114.wiki; fields and reading as in the layout above).
 *   x [T][H] bf16, w_router [E][H] bf16, router_bias f32 [E] or NULL (added to the
 *   selection score only).  given_topk i32 [T][k] or NULL: when non-NULL the selection is
 *   taken from it (each row k distinct experts in [0, E); a violation is reported as
 *   MOK_ERR_INVALID_ROUTING in the status word) and the gates are the router scores at
 *   those experts; x and w_router may then be NULL only if gates are not needed (pass
 *   gates = NULL too).
 *   Outputs (i32 unless noted): topk_idx [T][k], gates f32 [T][k] (nullable), counts [E],
 *   offsets [E+1], row_of [T*k], src_of [T*k].  ws: at least layout.ws_bytes.
 * The table is exact integer work: rows of an expert are in ascending assignment order. */
mok_status mok_schedule(const mok_layer_desc* desc, const void* x, const void* w_router,
                        const float* router_bias, const int32_t* given_topk, int32_t* topk_idx,
                        float* gates, int32_t* counts, int32_t* offsets, int32_t* row_of,
                        int32_t* src_of, void* ws, size_t ws_bytes, void* stream);

/* mok_schedule without a workspace (the pages have no counterpart of this entry point).
 * For callers that cannot allocate device memory when they route tokens: code running under
 * an allocator that forbids new allocations (a step whose memory plan is fixed), a runtime
 * that only hands out its own pre-sized buffers, or a plain C caller without a CUDA
 * allocator.  Same arguments, outputs and results as mok_schedule, minus ws / ws_bytes; the
 * scratch (status word and router logits) is one array compiled into the library:
 * MOK_NOALLOC_MAX_LOGITS floats plus 256 bytes (about 4 MiB), held in the memory of every
 * GPU that loads the library until the process exits.
 *   - Rejects T * E > MOK_NOALLOC_MAX_LOGITS with MOK_ERR_WORKSPACE_TOO_SMALL when the router
 *     runs (x and w_router given); the given_topk-only path has no size limit beyond
 *     mok_layer_desc's.
 *   - device_status: NULL, or a DEVICE buffer of 2 int32 that receives (code, site) of the
 *     first device-side error of this call, as mok_read_status would report it.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current); make that first call before any stream capture.
 *   - Every call on a device shares the array and it keeps the last call's contents (the
 *     status word is cleared at the start of each call).  Calls whose work overlaps on the
 *     GPU (other streams, other host threads) race on it: order them.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
#define MOK_NOALLOC_MAX_LOGITS (1 << 20)
mok_status mok_schedule_noalloc(const mok_layer_desc* desc, const void* x, const void* w_router,
                                const float* router_bias, const int32_t* given_topk, int32_t* topk_idx,
                                float* gates, int32_t* counts, int32_t* offsets, int32_t* row_of,
                                int32_t* src_of, int32_t* device_status, void* stream);

/* Layer forward: y [T][H] bf16 = sum over the k selected experts of gate * SwiGLU-FFN(x).
 *   w13 [E][2I][H] bf16 (rows 0..I-1 gate projection, I..2I-1 up projection),
 *   w2 [E][H][I] bf16, router_bias and given_topk as in mok_schedule.
 *   ctx (layout.ctx_bytes) receives what the backward needs; ws (layout.ws_bytes) is
 *   scratch and also holds the status word.  Pointers to x, weights, y, ctx and ws must be
 *   16-byte aligned (TMA).  MXFP8 is not accepted here (MOK_ERR_UNSUPPORTED).
 *   With ring_bytes > 0 the dispatched rows live only in the ring (ctx x_g is not written) and y
 *   is bitwise the same as without the ring.  The ring-based backward (mok_moe_backward on the
 *   same ctx and ws) reuses the minibatches the ring still holds and gathers again only those it
 *   overwrote ("Mixture-of-Kittens (MoK)", sd114.wiki, ring-buffer section); given another ws it
 *   gathers them all, with the same results.  The ring launch is cooperative: all of its CTAs
 *   must be resident at once (one per SM). */
mok_status mok_moe_forward(const mok_layer_desc* desc, const void* x, const void* w_router,
                           const float* router_bias, const int32_t* given_topk, const void* w13,
                           const void* w2, void* y, void* ctx, size_t ctx_bytes, void* ws,
                           size_t ws_bytes, void* stream);

/* IEEE fp16 copy of a bf16 tensor: dst [n] fp16 = src [n] bf16 rounded to nearest even (exact
 * for magnitudes 2^-14 .. 65504; smaller values become fp16 subnormals, larger ones infinities).
 * For the fp16 W2 of MOK_FLAG_W2_F16 (no counterpart on the pages: a precision choice of this
 * library for the tensor-bound GEMM2).  Device pointers, 16-byte aligned; async on `stream`. */
mok_status mok_convert_f16(const void* src, void* dst, int64_t n, void* stream);

/* MXFP8 weights for mok_moe_forward_mxfp8.  MXFP8 is one of the two precisions of the pages'
 * kernel ("Mixture-of-Kittens (MoK)", sd114.wiki, benchmark section); the format is read as OCP
 * Microscaling v1.0: E4M3 elements, one E8M0 scale per 32 consecutive elements along the GEMM's
 * reduction dimension, X = clamp(floor(log2 amax) - 8, -127, 127), elements RNE(v / 2^X)
 * saturated at +-448, scale byte X + 127.
 *   w13 [E][2I][H] bf16 -> w13_q [E][2I][H] E4M3 bytes, w13_scale [E][I/64][H/128][512] bytes
 *   w2  [E][H][I]  bf16 -> w2_q  [E][H][I]  E4M3 bytes, w2_scale  [E][H/128][I/128][512]  bytes
 * Scales come in 512-byte blocks, one per 128-row tile and 128-element stage of the reduction
 * dimension, in the order the tensor cores read them from tensor memory: row 32 j + l (of the
 * tile) and 32-element block b (of the stage) at byte 16 l + 4 j + b.  The 128-row tiles of W13
 * pair the gate rows 64 t .. 64 t + 63 (tile rows 0..63) with the up rows I + 64 t .. I + 64 t + 63
 * (tile rows 64..127): the rows one CTA of the SwiGLU GEMM multiplies.  All device pointers,
 * 16-byte aligned. */
mok_status mok_quantize_weights(const mok_layer_desc* desc, const void* w13, const void* w2, void* w13_q,
                                void* w13_scale, void* w2_q, void* w2_scale, void* stream);

/* Backward-direction MXFP8 weights for mok_moe_backward_mxfp8: each GEMM of the backward
 * quantises its operands along its own reduction dimension, so the weights are quantised again,
 * along the other axis, and stored transposed so that the reduction dimension is contiguous:
 *   w2  [E][H][I]  -> w2t_q  [E][I][H]  E4M3, quantised along H (for dA' = dY_g W2[e]),
 *                     w2t_scale [E][I/128][H/128][512]
 *   w13 [E][2I][H] -> w13t_q [E][H][2I] E4M3, quantised along 2I (for dX_g = dHU W13[e]),
 *                     w13t_scale [E][H/128][2I/128][512]
 * Scale blocks as for mok_quantize_weights (row 32 j + l of a 128-row tile and 32-element block b
 * of a 128-element stage at byte 16 l + 4 j + b).  Same rule as mok_quantize_weights.  All device
 * pointers, 16-byte aligned. */
mok_status mok_quantize_weights_backward(const mok_layer_desc* desc, const void* w13, const void* w2, void* w13t_q,
                                         void* w13t_scale, void* w2t_q, void* w2t_scale, void* stream);

/* Layer backward with MXFP8 expert GEMMs (desc->precision must be MOK_MXFP8), after
 * mok_moe_forward_mxfp8 with the same ctx.  Every expert GEMM operand is quantised in 32-element
 * blocks along that GEMM's reduction dimension: dY_g (gathered, along H) and W2 along H for dA';
 * dh|du along 2I and W13 along 2I for dX_g; for the weight gradients both operands along the
 * expert's rows (gate * dY and a for dW2, dh|du and the dispatched x for dW13), in 32-row blocks
 * that start at the expert's first row.  dA' and dX_g run on the FP8 tensor path (block-scaled MMAs
 * on the E4M3 weights of mok_quantize_weights_backward); the weight gradients multiply the exact
 * values of their quantised operands on the bf16 tensor path.  The gate gradient is <dA', a> in the
 * SwiGLU backward epilogue, with dA' the quantised product; the router backward and the reverse
 * dispatch are the bf16 path's.  Outputs and ws as for mok_moe_backward (ws layout from an MXFP8
 * descriptor). */
mok_status mok_moe_backward_mxfp8(const mok_layer_desc* desc, const void* dy, const void* x, const void* w_router,
                                  const void* w13t_q, const void* w13t_scale, const void* w2t_q, const void* w2t_scale,
                                  const void* ctx, size_t ctx_bytes, void* dx, float* dw_router, void* dw13, void* dw2,
                                  float* dgates, void* ws, size_t ws_bytes, void* stream);

/* Layer forward with MXFP8 expert GEMMs (desc->precision must be MOK_MXFP8, no ring).  As
 * mok_moe_forward, with the expert weights given as mok_quantize_weights output.  The MXFP8
 * activation quantisation sits on the data path ("把 MoE 通信延迟从 103μs 压到 18μs：Cursor 开源
 * GPU 内核 MoK", aientropygate.com, §03 ③): the gather quantises each dispatched row in
 * 32-element blocks along H and the GEMM1 epilogue quantises a = silu(h) * u along I, both into
 * E4M3 bytes and scale blocks (layout.mx_xq / mx_xsf, mx_aq / mx_asf in ws).  The expert GEMMs
 * run on the FP8 tensor path (block-scaled MMAs that apply the E8M0 scales themselves) and
 * accumulate in fp32.  The router stays in bf16.  ctx as for mok_moe_forward except that ctx x_g
 * is not written (the MXFP8 backward takes the dispatched rows from x).  The MXFP8 backward is
 * mok_moe_backward_mxfp8; mok_moe_backward returns MOK_ERR_UNSUPPORTED for an MXFP8 descriptor. */
mok_status mok_moe_forward_mxfp8(const mok_layer_desc* desc, const void* x, const void* w_router,
                                 const float* router_bias, const int32_t* given_topk, const void* w13_q,
                                 const void* w13_scale, const void* w2_q, const void* w2_scale, void* y,
                                 void* ctx, size_t ctx_bytes, void* ws, size_t ws_bytes, void* stream);

/* Layer backward for upstream gradient dy [T][H] bf16, using the ctx written by the
 * matching mok_moe_forward (same desc, inputs and weights).  Outputs:
 *   dx [T][H] bf16, dw_router [E][H] f32, dw13 [E][2I][H] and dw2 [E][H][I] in f32 (bf16
 *   with MOK_FLAG_WGRAD_BF16), dgates [T][k] f32 (nullable): gradient w.r.t. each gate.
 *   An expert that received no rows gets an all-zero weight gradient.
 * The selection is held fixed; the router bias gets no gradient.  The gate gradient
 * <dA', a> of each row is formed in the SwiGLU-backward epilogue (the router-weight
 * gradient "fused into the SwiGLU backward" of the pages' benchmark section). */
mok_status mok_moe_backward(const mok_layer_desc* desc, const void* dy, const void* x,
                            const void* w_router, const void* w13, const void* w2,
                            const void* ctx, size_t ctx_bytes, void* dx, float* dw_router,
                            void* dw13, void* dw2, float* dgates, void* ws, size_t ws_bytes,
                            void* stream);

/* Synchronises `stream`, copies the device status word out of ws into
 * device_status[0] (code, a mok_status value) and device_status[1] (site), then clears it.
 * Host-blocking; not for use inside captured graphs. */
mok_status mok_read_status(void* ws, size_t ws_bytes, void* stream, int32_t* device_status);

/* Test hook for the bounded waits (no counterpart on the pages): launches one kernel
 * whose single thread waits on an mbarrier that nothing will complete, with the given
 * limit in milliseconds; the wait gives up, records MOK_ERR_TIMEOUT in the status word
 * of ws and the kernel returns normally.  Used to show that a stuck wait ends cleanly. */
mok_status mok_test_bounded_wait(void* ws, size_t ws_bytes, int32_t limit_ms, void* stream);

/* Per-kernel timing (tracing; no counterpart on the pages).  mok_trace_start enables it
 * for the whole process: every kernel the library launches from then on is bracketed by
 * two CUDA events recorded on the stream it is launched on, up to max_launches launches.
 * mok_trace_stop synchronises those events, sums the elapsed time per kernel name into
 * out[0..cap) (names in launch order of first appearance), stores the number of entries in
 * *n_out, frees the events and disables tracing.  Host-side state only; not thread-safe;
 * do not start it while a stream capture is active. */
typedef struct {
  char name[32];
  int32_t launches;
  float total_ms;
} mok_trace_entry;

mok_status mok_trace_start(int32_t max_launches);
mok_status mok_trace_stop(mok_trace_entry* out, int32_t cap, int32_t* n_out);

/* Human-readable name of a status code. */
const char* mok_status_string(mok_status s);

/* Number of SMs of the current device and the minimum minibatch (rows) whose expert-
 * grouped GEMM1 fills two full SM waves of 128x256 output tiles: ceil(2*n_sm*128*256/(2I)).
 * The pages state the two-wave rule and its result, 2,368 tokens, for hidden 7168 and
 * intermediate 2048 ("Mixture-of-Kittens (MoK)", sd114.wiki, overlap-granularity section;
 * aientropygate.com, §03 ②) but no formula; this is the reading that reproduces it for
 * 148 SMs.  n_sm <= 0 means: query the current device. */
int32_t mok_min_minibatch(int32_t n_sm, int32_t I);

#ifdef __cplusplus
}
#endif

#endif /* MOK_H_ */
