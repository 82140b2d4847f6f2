// C ABI of the layer (include/mok.h): argument checks, ctx / ws layout, and the launch
// sequences of the forward and backward passes.  No allocation, no host synchronisation
// in the compute calls; every kernel is enqueued on the caller's stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "kernels.cuh"
#include "mok.h"
#include "mx_tiles.h"

namespace {

constexpr int kMaxDevices = 64;

int sm_count() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mok_status check_desc(const mok_layer_desc* d) {
  if (d == nullptr) return MOK_ERR_INVALID_ARG;
  if (d->T < 1 || d->H < 1 || d->I < 1 || d->E < 1 || d->k < 1) return MOK_ERR_INVALID_ARG;
  if (d->k > d->E) return MOK_ERR_INVALID_ARG;
  if (d->router != MOK_ROUTER_SOFTMAX && d->router != MOK_ROUTER_SIGMOID) return MOK_ERR_INVALID_ARG;
  if (d->precision != MOK_BF16 && d->precision != MOK_MXFP8) return MOK_ERR_INVALID_ARG;
  if (!std::isfinite(d->route_scale)) return MOK_ERR_INVALID_ARG;
  if (d->minibatch < 0 || d->ring_bytes < 0) return MOK_ERR_INVALID_ARG;
  if ((d->flags & MOK_FLAG_GEMM_PAIR) && (d->flags & MOK_FLAG_GEMM_SINGLE)) return MOK_ERR_INVALID_ARG;
  // 128: one CTA's weight rows (half a CTA pair's 256-row tile) and the MXFP8 kernels' K step; a
  // pair tile over H or I that reaches past the end reads zeros there and stores none of it
  if (d->H % 128 != 0 || d->I % 128 != 0) return MOK_ERR_UNSUPPORTED;
  if (d->E > 1024 || d->k > 16) return MOK_ERR_UNSUPPORTED;
  const int64_t R = int64_t(d->T) * d->k;
  const int64_t width = d->H > 2 * d->I ? d->H : 2 * int64_t(d->I);
  if (R * width >= (int64_t(1) << 31)) return MOK_ERR_UNSUPPORTED;
  return MOK_OK;
}

// Expert GEMM kernels: by default the narrow-segment pair kernel (the expert's rows are the
// MMA's N, padded to 16 rows instead of a 128-row tile); MOK_FLAG_GEMM_SINGLE / MOK_FLAG_GEMM_PAIR
// ask for the row-tile kernels (dX_g has no pair row-tile form and runs on single CTAs then).
enum ExpertGemm { GEMM1 = 0, GEMM2 = 1, DGRAD_X = 2 };
// Weight gradients on CTA pairs (256 x 256 tiles) unless the row-tile kernels are asked for.
bool wgrad_pairs(const mok_layer_desc* d) { return (d->flags & (MOK_FLAG_GEMM_SINGLE | MOK_FLAG_GEMM_PAIR)) == 0; }
int gemm_variant(const mok_layer_desc* d, int which) {
  if (d->flags & MOK_FLAG_GEMM_PAIR) return which == DGRAD_X ? mok::GEMM_ROWS_SINGLE : mok::GEMM_ROWS_PAIR;
  if (d->flags & MOK_FLAG_GEMM_SINGLE) return mok::GEMM_ROWS_SINGLE;
  return mok::GEMM_NARROW;
}

// Two full waves of 128 x 256 GEMM1 output tiles over n_sm SMs, in rows: GEMM1 has 2I columns.
int32_t min_minibatch_rows(int n_sm, int I) {
  if (n_sm <= 0 || I <= 0) return 0;
  return static_cast<int32_t>((2LL * n_sm * 128 * 256 + 2LL * I - 1) / (2LL * I));
}

// Ring forward geometry: rows per minibatch m, minibatches n_mb, ring slots (minibatches the
// ring holds, at most n_mb).
struct RingGeom {
  int m = 0, n_mb = 0, slots = 0;
};

// Byte offset of the ring stamp (u64 [2]) after the [2][n_mb] i32 counters.
// counters: gathered [n_mb], consumed [n_mb], the GEMM1 tile ticket, the GEMM2 tile ticket and the
// GEMM2 epilogue count of the persistent ring forward; then the stamp, 16-byte aligned
int64_t ring_counter_ints(int n_mb) { return int64_t(2) * n_mb + 3; }
int64_t ring_stamp_offset(int n_mb) { return (ring_counter_ints(n_mb) * 4 + 15) & ~int64_t(15); }

mok_status ring_geometry(const mok_layer_desc* d, RingGeom* g) {
  const int64_t R = int64_t(d->T) * d->k;
  int64_t m = d->minibatch;
  if (m == 0) {
    m = min_minibatch_rows(sm_count(), d->I);
    if (m <= 0) return MOK_ERR_INVALID_ARG;  // no device to size the default minibatch
  }
  if (m > R) m = R;
  const int64_t n_mb = (R + m - 1) / m;
  int64_t slots = d->ring_bytes / (m * d->H * 2);
  if (slots < 1) return MOK_ERR_UNSUPPORTED;  // the ring must hold one minibatch
  if (slots > n_mb) slots = n_mb;
  g->m = (int)m;
  g->n_mb = (int)n_mb;
  g->slots = (int)slots;
  return MOK_OK;
}

mok_status fill_layout(const mok_layer_desc* d, mok_layout* L) {
  const int64_t T = d->T, H = d->H, I = d->I, E = d->E, k = d->k, R = T * k;
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L->topk_idx = take(T * k * 4);
  L->gates = take(T * k * 4);
  L->scores = take(T * E * 4);
  L->counts = take(E * 4);
  L->offsets = take((E + 1) * 4);
  L->row_of = take(R * 4);
  L->src_of = take(R * 4);
  L->tile_off = take((E + 1) * 4);
  L->gate_row = take(R * 4);
  L->x_g = take(R * H * 2);
  L->hu = take(R * 2 * I * 4);
  RingGeom rgeom;
  if (d->ring_bytes > 0) {
    const mok_status s = ring_geometry(d, &rgeom);
    if (s != MOK_OK) return s;
  }
  L->ring_stamp = d->ring_bytes > 0 ? take(16) : -1;
  L->ctx_bytes = off;
  off = 0;
  L->status = take(mok::STATUS_BYTES);
  L->logits = take(T * E * 4);
  L->sched = take(int64_t(mok::schedule_blocks((int)R)) * E * 4);
  L->act = take(R * I * 2);
  L->act_lo = take(R * I * 2);
  L->expert_out = take(R * H * 4);
  L->dy_g = take(R * H * 2);
  L->dhu = take(R * 2 * I * 2);
  L->dhu_lo = take(R * 2 * I * 2);
  L->gact = take(R * I * 2);
  L->gact_lo = take(R * I * 2);
  L->dx_g = take(R * H * 4);
  L->dg_part = take(R * (I / 128) * 4);
  L->dlogits = take(T * E * 4);
  L->ring = L->mb_tables = L->mb_counters = -1;
  if (d->ring_bytes > 0) {
    const RingGeom& g = rgeom;
    // the dispatched rows of every minibatch; the token ring is the last slots * m of them
    L->ring = take(int64_t(g.n_mb) * g.m * H * 2);
    // mb_off [n_mb][E+1], mb_toff [n_mb][E+1], mb_tiles [n_mb], mb_start [n_mb+1]
    L->mb_tables = take((int64_t(2) * g.n_mb * (E + 1) + 2 * int64_t(g.n_mb) + 1) * 4);
    // counters [2][n_mb] and the tile ticket, then the u64 [2] stamp of the forward that filled the ring
    L->mb_counters = take(ring_stamp_offset(g.n_mb) + 16);
  }
  L->mx_dhu_r = L->mx_xg_r = L->mx_do_r = L->mx_a_r = L->mx_blk_off = -1;
  L->mx_xq = L->mx_xsf = L->mx_aq = L->mx_asf = L->mx_dyq = L->mx_dysf = L->mx_dhuq = L->mx_dhusf = -1;
  if (d->precision == MOK_MXFP8) {
    L->mx_dhu_r = take(R * 2 * I * 2);
    L->mx_xg_r = take(R * H * 2);
    L->mx_do_r = take(R * H * 2);
    L->mx_a_r = take(R * I * 2);
    L->mx_blk_off = take((E + 1) * 4);
    const int64_t RP = mok::mx_rows_padded_bound(R, (int)E), G = mok::mx_row_groups(R, (int)E);
    L->mx_xq = take(RP * H);
    L->mx_xsf = take(G * (H / mok::MX_BK) * mok::MX_SF_BLOCK);
    L->mx_aq = take(RP * I);
    L->mx_asf = take(G * (I / mok::MX_BK) * mok::MX_SF_BLOCK);
    L->mx_dyq = take(RP * H);
    L->mx_dysf = take(G * (H / mok::MX_BK) * mok::MX_SF_BLOCK);
    L->mx_dhuq = take(RP * 2 * I);
    L->mx_dhusf = take(G * (2 * I / mok::MX_BK) * mok::MX_SF_BLOCK);
  }
  L->ws_bytes = off;
  return MOK_OK;
}

template <typename T>
T* at(void* base, int64_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}
template <typename T>
const T* at(const void* base, int64_t off) {
  return reinterpret_cast<const T*>(static_cast<const char*>(base) + off);
}

#define MOK_CUDA(call)                       \
  do {                                       \
    if ((call) != cudaSuccess) return MOK_ERR_CUDA; \
  } while (0)

// ------------------------------------------------------------------ per-kernel trace
struct TraceRec {
  const char* name;
  cudaEvent_t start, stop;
};

struct Trace {
  std::mutex mu;
  bool on = false;
  int cap = 0;
  int used = 0;
  TraceRec* recs = nullptr;
} g_trace;

// Records a start event before and a stop event after the launch `call` on stream `st`.
template <typename F>
cudaError_t traced(const char* name, cudaStream_t st, F&& call) {
  TraceRec* rec = nullptr;
  if (g_trace.on) {
    std::lock_guard<std::mutex> lock(g_trace.mu);
    if (g_trace.on && g_trace.used < g_trace.cap) {
      rec = &g_trace.recs[g_trace.used++];
      rec->name = name;
    }
  }
  if (rec) cudaEventRecord(rec->start, st);
  const cudaError_t err = call();
  if (rec) cudaEventRecord(rec->stop, st);
  return err;
}

#define MOK_LAUNCH(name, st, expr) MOK_CUDA(traced(name, st, [&] { return (expr); }))

}  // namespace

extern "C" {

const char* mok_status_string(mok_status s) {
  switch (s) {
    case MOK_OK: return "ok";
    case MOK_ERR_INVALID_ARG: return "invalid argument";
    case MOK_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case MOK_ERR_WORKSPACE_TOO_SMALL: return "workspace or ctx too small";
    case MOK_ERR_CUDA: return "CUDA error";
    case MOK_ERR_TIMEOUT: return "device wait timed out";
    case MOK_ERR_INVALID_ROUTING: return "invalid routing (expert index out of range or repeated)";
  }
  return "unknown status";
}

mok_status mok_get_layout(const mok_layer_desc* desc, mok_layout* layout) {
  if (layout == nullptr) return MOK_ERR_INVALID_ARG;
  const mok_status s = check_desc(desc);
  if (s != MOK_OK) return s;
  return fill_layout(desc, layout);
}

mok_status mok_workspace_size(const mok_layer_desc* desc, size_t* ws_bytes, size_t* ctx_bytes) {
  if (ws_bytes == nullptr || ctx_bytes == nullptr) return MOK_ERR_INVALID_ARG;
  mok_layout L;
  const mok_status s = mok_get_layout(desc, &L);
  if (s != MOK_OK) return s;
  *ws_bytes = (size_t)L.ws_bytes;
  *ctx_bytes = (size_t)L.ctx_bytes;
  return MOK_OK;
}

int32_t mok_min_minibatch(int32_t n_sm, int32_t I) {
  if (n_sm <= 0) n_sm = sm_count();
  return min_minibatch_rows(n_sm, I);
}

mok_status mok_schedule(const mok_layer_desc* d, const void* x, const void* w_router, const float* router_bias,
                        const int32_t* given_topk, int32_t* topk_idx, float* gates, int32_t* counts,
                        int32_t* offsets, int32_t* row_of, int32_t* src_of, void* ws, size_t ws_bytes,
                        void* stream) {
  mok_status s = check_desc(d);
  if (s != MOK_OK) return s;
  mok_layout L;
  s = fill_layout(d, &L);
  if (s != MOK_OK) return s;
  if (!topk_idx || !counts || !offsets || !row_of || !src_of || !ws) return MOK_ERR_INVALID_ARG;
  if ((int64_t)ws_bytes < L.ws_bytes) return MOK_ERR_WORKSPACE_TOO_SMALL;
  const bool have_router = x != nullptr && w_router != nullptr;
  if (!have_router && (given_topk == nullptr || gates != nullptr)) return MOK_ERR_INVALID_ARG;
  if (have_router && (!aligned16(x) || !aligned16(w_router))) return MOK_ERR_INVALID_ARG;
  const int n_sm = sm_count();
  if (n_sm <= 0) return MOK_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = at<int>(ws, L.status);
  float* logits = at<float>(ws, L.logits);
  MOK_CUDA(cudaMemsetAsync(status, 0, mok::STATUS_BYTES, st));
  if (have_router) MOK_LAUNCH("router_gemm", st, mok::launch_router_gemm(x, w_router, d->T, d->H, d->E, logits, status, n_sm, st));
  MOK_LAUNCH("topk", st, mok::launch_topk(have_router ? logits : nullptr, router_bias, given_topk, d->T, d->E, d->k, d->router,
                            d->renorm, d->route_scale, topk_idx, gates, nullptr, status, st));
  MOK_LAUNCH("schedule", st, mok::launch_schedule_multi(topk_idx, nullptr, d->T * d->k, d->E, counts, offsets, row_of,
                                                        src_of, nullptr, nullptr, at<int32_t>(ws, L.sched), status, st));
  return MOK_OK;
}

mok_status mok_moe_forward(const mok_layer_desc* d, const void* x, const void* w_router, const float* router_bias,
                           const int32_t* given_topk, const void* w13, const void* w2, void* y, void* ctx,
                           size_t ctx_bytes, void* ws, size_t ws_bytes, void* stream) {
  mok_status s = check_desc(d);
  if (s != MOK_OK) return s;
  if (d->precision != MOK_BF16) return MOK_ERR_UNSUPPORTED;
  if (!x || !w_router || !w13 || !w2 || !y || !ctx || !ws) return MOK_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w13) || !aligned16(w2) || !aligned16(y) ||
      !aligned16(ctx) || !aligned16(ws))
    return MOK_ERR_INVALID_ARG;
  mok_layout L;
  s = fill_layout(d, &L);
  if (s != MOK_OK) return s;
  if ((int64_t)ctx_bytes < L.ctx_bytes || (int64_t)ws_bytes < L.ws_bytes) return MOK_ERR_WORKSPACE_TOO_SMALL;
  const int n_sm = sm_count();
  if (n_sm <= 0) return MOK_ERR_CUDA;
  // fp16 W2 (MOK_FLAG_W2_F16): the narrow-segment GEMMs without the ring only
  const bool w2_f16 = (d->flags & MOK_FLAG_W2_F16) != 0;
  if (w2_f16 && (d->ring_bytes > 0 || gemm_variant(d, GEMM2) != mok::GEMM_NARROW)) return MOK_ERR_UNSUPPORTED;
  // the ring forward in one persistent launch (narrow GEMMs, top-k of at most 8)
  const bool ring_persistent = d->ring_bytes > 0 && (d->flags & MOK_FLAG_RING_PERSISTENT) != 0 &&
                               gemm_variant(d, GEMM1) == mok::GEMM_NARROW && d->k <= 8;
  RingGeom rg;
  const int comm = d->comm_sms > 0 ? d->comm_sms : 12;
  if (d->ring_bytes > 0) {
    s = ring_geometry(d, &rg);
    if (s != MOK_OK) return s;
    if (comm >= n_sm) return MOK_ERR_INVALID_ARG;
    // the CTA-pair ring kernel takes its gathering CTAs in whole clusters of two
    if (gemm_variant(d, GEMM1) == mok::GEMM_NARROW && comm % 2 != 0) return MOK_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = d->T, H = d->H, I = d->I, E = d->E, k = d->k, R = T * k;
  int* status = at<int>(ws, L.status);
  int32_t* topk_idx = at<int32_t>(ctx, L.topk_idx);
  float* gates = at<float>(ctx, L.gates);
  int32_t* offsets = at<int32_t>(ctx, L.offsets);
  int32_t* tile_off = at<int32_t>(ctx, L.tile_off);
  int32_t* row_of = at<int32_t>(ctx, L.row_of);
  int32_t* src_of = at<int32_t>(ctx, L.src_of);
  void* x_g = at<char>(ctx, L.x_g);
  float* hu = at<float>(ctx, L.hu);
  void* act = at<char>(ws, L.act);
  void* act_lo = at<char>(ws, L.act_lo);
  float* o = at<float>(ws, L.expert_out);
  float* logits = at<float>(ws, L.logits);

  MOK_CUDA(cudaMemsetAsync(status, 0, mok::STATUS_BYTES, st));
  // 1. router logits x W_r^T (tensor cores, fp32 accumulate)
  MOK_LAUNCH("router_gemm", st, mok::launch_router_gemm(x, w_router, T, H, E, logits, status, n_sm, st));
  // 2. scores, top-k and gates
  MOK_LAUNCH("topk", st, mok::launch_topk(logits, router_bias, given_topk, T, E, k, d->router, d->renorm, d->route_scale,
                            topk_idx, gates, at<float>(ctx, L.scores), status, st));
  // 3. schedule table
  MOK_LAUNCH("schedule", st, mok::launch_schedule_multi(topk_idx, gates, R, E, at<int32_t>(ctx, L.counts), offsets, row_of,
                                                        src_of, tile_off, at<float>(ctx, L.gate_row),
                                                        at<int32_t>(ws, L.sched), status, st));
  if (d->ring_bytes == 0) {
    // 4. pull dispatch into expert-contiguous rows
    MOK_LAUNCH("gather_x", st, mok::launch_gather_rows(x, src_of, k, R, H, x_g, n_sm, st));
    // 5. grouped GEMM1 with the SwiGLU epilogue
    MOK_LAUNCH("gemm1_swiglu", st, mok::launch_gemm1_swiglu(x_g, w13, R, H, I, E, offsets, tile_off, hu, act, act_lo,
                                                            status, n_sm, gemm_variant(d, GEMM1), w2_f16, st));
  } else {
    // 4-5. ring forward: per-minibatch tables, then one persistent launch in which `comm`
    //      CTAs gather minibatches into the ring while the others run GEMM1 on them
    int32_t* tab = at<int32_t>(ws, L.mb_tables);
    int32_t* mb_off = tab;
    int32_t* mb_toff = mb_off + (size_t)rg.n_mb * (E + 1);
    int32_t* mb_tiles = mb_toff + (size_t)rg.n_mb * (E + 1);
    int32_t* mb_start = mb_tiles + rg.n_mb;
    int32_t* counters = at<int32_t>(ws, L.mb_counters);
    const int ring_variant = gemm_variant(d, GEMM1);
    MOK_LAUNCH("ring_tables", st,
               mok::launch_mb_tables(offsets, E, R, rg.m, rg.n_mb, mok::ring_tiles_per_chunk(ring_variant, R, E, I),
                                     mok::ring_chunk_rows(ring_variant), mb_off,
                                     mb_toff, mb_tiles, mb_start, st));
    MOK_CUDA(cudaMemsetAsync(counters, 0, sizeof(int32_t) * ring_counter_ints(rg.n_mb), st));
    mok::RingArgs ra;
    ra.x = x;
    ra.src_of = src_of;
    ra.k = k;
    ra.R = R;
    ra.H = H;
    ra.I = I;
    ra.E = E;
    ra.mb_rows = rg.m;
    ra.n_mb = rg.n_mb;
    ra.ring_slots = rg.slots;
    // minibatch mb in slot (mb + shift) % slots: the last `slots` minibatches, which the ring still
    // holds after the forward, then sit in slot order at their own rows of the dispatched-row region
    ra.ring_shift = (rg.slots - rg.n_mb % rg.slots) % rg.slots;
    ra.comm_ctas = comm;
    ra.ring = at<char>(ws, L.ring) + (int64_t)(rg.n_mb - rg.slots) * rg.m * H * 2;
    ra.mb_off = mb_off;
    ra.mb_toff = mb_toff;
    ra.mb_start = mb_start;
    ra.gathered = counters;
    ra.consumed = counters + rg.n_mb;
    ra.ticket = counters + 2 * rg.n_mb;
    ra.ticket2 = counters + 2 * rg.n_mb + 1;
    ra.done = counters + 2 * rg.n_mb + 2;
    if (ring_persistent) {
      // one launch for the rest of the forward: gather, GEMM1 + SwiGLU, GEMM2, weighted merge
      MOK_LAUNCH("ring_forward", st,
                 mok::launch_ring_forward(ra, w13, w2, hu, act, act_lo, o, gates, row_of, T, y, status, n_sm, st));
    } else {
      MOK_LAUNCH("ring_gemm1_swiglu", st,
                 mok::launch_ring_gemm1(ra, w13, hu, act, act_lo, status, n_sm, ring_variant, st));
    }
    // the ring rows are this forward's (the backward reuses them when it is given this ws)
    MOK_LAUNCH("ring_stamp", st,
               mok::launch_ring_stamp(at<unsigned long long>(ctx, L.ring_stamp),
                                      reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(counters) +
                                                                            ring_stamp_offset(rg.n_mb)),
                                      (unsigned long long)reinterpret_cast<uintptr_t>(ctx), st));
  }
  if (ring_persistent) return MOK_OK;
  // 6. grouped GEMM2 (a as hi + lo, or as fp16 against the fp16 W2), fp32 expert outputs
  MOK_LAUNCH("gemm2", st,
             mok::launch_gemm2(act, act_lo, w2, R, H, I, E, offsets, tile_off, o, status, n_sm,
                               gemm_variant(d, GEMM2), w2_f16, st));
  // 7. weighted merge in fixed order
  MOK_LAUNCH("combine", st, mok::launch_combine(o, gates, row_of, T, k, H, nullptr, nullptr, nullptr, E, 0, y, n_sm, st));
  return MOK_OK;
}

mok_status mok_convert_f16(const void* src, void* dst, int64_t n, void* stream) {
  if (!src || !dst || n < 0 || !aligned16(src) || !aligned16(dst)) return MOK_ERR_INVALID_ARG;
  if (n == 0) return MOK_OK;
  const int n_sm = sm_count();
  if (n_sm <= 0) return MOK_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOK_LAUNCH("convert_f16", st, mok::launch_bf16_to_f16(src, dst, n, n_sm, st));
  return MOK_OK;
}

mok_status mok_quantize_weights(const mok_layer_desc* d, const void* w13, const void* w2, void* w13_q, void* w13_scale,
                                void* w2_q, void* w2_scale, void* stream) {
  mok_status s = check_desc(d);
  if (s != MOK_OK) return s;
  const void* ptrs[] = {w13, w2, w13_q, w13_scale, w2_q, w2_scale};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return MOK_ERR_INVALID_ARG;
  const int n_sm = sm_count();
  if (n_sm <= 0) return MOK_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOK_LAUNCH("quantize_w13", st,
             mok::launch_quantize_weights(w13, w13_q, w13_scale, d->E, 2 * d->I, d->H, d->I, n_sm, st));
  MOK_LAUNCH("quantize_w2", st, mok::launch_quantize_weights(w2, w2_q, w2_scale, d->E, d->H, d->I, 0, n_sm, st));
  return MOK_OK;
}

mok_status mok_quantize_weights_backward(const mok_layer_desc* d, const void* w13, const void* w2, void* w13t_q,
                                         void* w13t_scale, void* w2t_q, void* w2t_scale, void* stream) {
  mok_status s = check_desc(d);
  if (s != MOK_OK) return s;
  const void* ptrs[] = {w13, w2, w13t_q, w13t_scale, w2t_q, w2t_scale};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return MOK_ERR_INVALID_ARG;
  const int n_sm = sm_count();
  if (n_sm <= 0) return MOK_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int H = d->H, I = d->I, E = d->E;
  // W2[e] [H][I] -> [I][H] quantised along H; W13[e] [2I][H] -> [H][2I] quantised along 2I
  MOK_LAUNCH("quantize_w2_bwd", st, mok::launch_quantize_transpose(w2, w2t_q, w2t_scale, E, H, I, n_sm, st));
  MOK_LAUNCH("quantize_w13_bwd", st, mok::launch_quantize_transpose(w13, w13t_q, w13t_scale, E, 2 * I, H, n_sm, st));
  return MOK_OK;
}

mok_status mok_moe_backward_mxfp8(const mok_layer_desc* d, const void* dy, const void* x, const void* w_router,
                                  const void* w13t_q, const void* w13t_scale, const void* w2t_q, const void* w2t_scale,
                                  const void* ctx, size_t ctx_bytes, void* dx, float* dw_router, void* dw13, void* dw2,
                                  float* dgates, void* ws, size_t ws_bytes, void* stream) {
  mok_status s = check_desc(d);
  if (s != MOK_OK) return s;
  if (d->precision != MOK_MXFP8 || d->ring_bytes != 0) return MOK_ERR_UNSUPPORTED;
  const void* ptrs[] = {dy, x, w_router, w13t_q, w13t_scale, w2t_q, w2t_scale, ctx, dx, dw_router, dw13, dw2, ws};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return MOK_ERR_INVALID_ARG;
  mok_layout L;
  s = fill_layout(d, &L);
  if (s != MOK_OK) return s;
  if ((int64_t)ctx_bytes < L.ctx_bytes || (int64_t)ws_bytes < L.ws_bytes) return MOK_ERR_WORKSPACE_TOO_SMALL;
  const int n_sm = sm_count();
  if (n_sm <= 0) return MOK_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = d->T, H = d->H, I = d->I, E = d->E, k = d->k, R = T * k;
  const int RP = (int)mok::mx_rows_padded_bound(R, E), G = (int)mok::mx_row_groups(R, E);
  int* status = at<int>(ws, L.status);
  // the work counters of this call start at zero (the status word keeps what the forward left)
  MOK_CUDA(cudaMemsetAsync(status + mok::STATUS_COUNTERS, 0, mok::STATUS_BYTES - 4 * mok::STATUS_COUNTERS, st));
  const int32_t* topk_idx = at<int32_t>(ctx, L.topk_idx);
  const float* gates = at<float>(ctx, L.gates);
  const float* scores = at<float>(ctx, L.scores);
  const int32_t* offsets = at<int32_t>(ctx, L.offsets);
  const int32_t* row_of = at<int32_t>(ctx, L.row_of);
  const int32_t* src_of = at<int32_t>(ctx, L.src_of);
  const float* gate_row = at<float>(ctx, L.gate_row);
  const float* hu = at<float>(ctx, L.hu);
  void* dhu = at<char>(ws, L.dhu);
  void* dhu_lo = at<char>(ws, L.dhu_lo);
  float* dx_g = at<float>(ws, L.dx_g);
  float* dg_part = at<float>(ws, L.dg_part);
  float* dl = at<float>(ws, L.dlogits);
  void* dhu_r = at<char>(ws, L.mx_dhu_r);
  void* xg_r = at<char>(ws, L.mx_xg_r);
  void* do_r = at<char>(ws, L.mx_do_r);
  void* a_r = at<char>(ws, L.mx_a_r);
  int32_t* blk_off = at<int32_t>(ws, L.mx_blk_off);
  void* dyq = at<char>(ws, L.mx_dyq);
  void* dysf = at<char>(ws, L.mx_dysf);
  void* dhuq = at<char>(ws, L.mx_dhuq);
  void* dhusf = at<char>(ws, L.mx_dhusf);
  const int wgrad_f32 = (d->flags & MOK_FLAG_WGRAD_BF16) ? 0 : 1;

  // 1. reverse combine: dY rows gathered into the padded row space, quantised along H (the reduction
  //    dimension of dA') into E4M3 bytes and scale blocks
  MOK_LAUNCH("mx_block_offsets", st, mok::launch_mx_block_offsets(offsets, E, blk_off, st));
  MOK_LAUNCH("gather_dy_mx", st, mok::launch_gather_rows_mxf8(dy, src_of, topk_idx, offsets, blk_off, k, R, H, E, dyq,
                                                              dysf, st));
  // 2. dA' = dY_g W2[e] on the FP8 tensor path (W2 stored [I][H], quantised along H); SwiGLU backward
  //    epilogue: dh | du (bf16 hi / lo, and E4M3 along 2I for dX_g) and the partial gate gradients
  //    <dA', a> per 128 intermediate indices
  MOK_LAUNCH("dgrad_swiglu_mx", st,
             mok::launch_dgrad_swiglu_mxf8(dyq, dysf, w2t_q, w2t_scale, RP, G, R, H, I, E, offsets, blk_off, hu,
                                           gate_row, dhu, dhu_lo, dhuq, dhusf, dg_part, status, n_sm, st));
  // 3. the weight-gradient operands, each quantised along the expert's rows (its reduction)
  MOK_LAUNCH("mx_dhu_rows", st, mok::launch_mx_quant_rows(1, R, 2 * I, E, 0, offsets, blk_off, dhu, dhu_lo, nullptr,
                                                          nullptr, nullptr, k, dhu_r, n_sm, st));
  MOK_LAUNCH("mx_xg_rows", st, mok::launch_mx_quant_rows(3, R, H, E, 0, offsets, blk_off, x, nullptr, nullptr, nullptr,
                                                         src_of, k, xg_r, n_sm, st));
  MOK_LAUNCH("mx_do_rows", st, mok::launch_mx_quant_rows(4, R, H, E, 0, offsets, blk_off, dy, nullptr, nullptr,
                                                         gate_row, src_of, k, do_r, n_sm, st));
  MOK_LAUNCH("mx_a_rows", st, mok::launch_mx_quant_rows(2, R, I, E, 0, offsets, blk_off, nullptr, nullptr, hu, nullptr,
                                                        nullptr, k, a_r, n_sm, st));
  // 4. dX_g = dHU W13[e] on the FP8 tensor path (W13 stored [H][2I], quantised along 2I)
  MOK_LAUNCH("dgrad_x_mx", st, mok::launch_dgrad_x_mxf8(dhuq, dhusf, w13t_q, w13t_scale, RP, G, R, H, I, E, offsets,
                                                        blk_off, dx_g, status, n_sm, st));
  // 5. dW2[e] = (g dY)^T a stored as [H][I]; dW13[e] = dHU^T x_g stored as [2I][H] (exact products of the
  //    quantised values on the bf16 kernels)
  MOK_LAUNCH("wgrad_w2", st, mok::launch_wgrad(a_r, nullptr, I, do_r, nullptr, H, R, E, offsets, dw2, wgrad_f32, status,
                                               status + mok::STATUS_COUNTERS + mok::CNT_WGRAD_W2, wgrad_pairs(d),
                                               n_sm, st));
  MOK_LAUNCH("wgrad_w13", st, mok::launch_wgrad(xg_r, nullptr, H, dhu_r, nullptr, 2 * I, R, E, offsets, dw13,
                                                wgrad_f32, status,
                                                status + mok::STATUS_COUNTERS + mok::CNT_WGRAD_W13, wgrad_pairs(d),
                                                n_sm, st));
  // 6-8. gate and router gradients, router weight gradient, reverse dispatch (as in bf16)
  MOK_LAUNCH("router_dlogits", st, mok::launch_router_dlogits(dg_part, I / 128, row_of, topk_idx, gates, scores, T, E, k,
                                                              d->router, d->renorm, d->route_scale, dgates, dl, st));
  MOK_LAUNCH("router_wgrad", st, mok::launch_router_wgrad(dl, x, offsets, src_of, T, H, E, k,
                                                          d->router == MOK_ROUTER_SIGMOID ? 1 : 0, dw_router, st));
  MOK_LAUNCH("combine_dx", st, mok::launch_combine(dx_g, nullptr, row_of, T, k, H, dl, w_router, topk_idx, E,
                                                   d->router == MOK_ROUTER_SOFTMAX ? 1 : 0, dx, n_sm, st));
  return MOK_OK;
}

mok_status mok_moe_forward_mxfp8(const mok_layer_desc* d, const void* x, const void* w_router,
                                 const float* router_bias, const int32_t* given_topk, const void* w13_q,
                                 const void* w13_scale, const void* w2_q, const void* w2_scale, void* y, void* ctx,
                                 size_t ctx_bytes, void* ws, size_t ws_bytes, void* stream) {
  mok_status s = check_desc(d);
  if (s != MOK_OK) return s;
  if (d->precision != MOK_MXFP8 || d->ring_bytes != 0) return MOK_ERR_UNSUPPORTED;
  const void* ptrs[] = {x, w_router, w13_q, w13_scale, w2_q, w2_scale, y, ctx, ws};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return MOK_ERR_INVALID_ARG;
  mok_layout L;
  s = fill_layout(d, &L);
  if (s != MOK_OK) return s;
  if ((int64_t)ctx_bytes < L.ctx_bytes || (int64_t)ws_bytes < L.ws_bytes) return MOK_ERR_WORKSPACE_TOO_SMALL;
  const int n_sm = sm_count();
  if (n_sm <= 0) return MOK_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = d->T, H = d->H, I = d->I, E = d->E, k = d->k, R = T * k;
  int* status = at<int>(ws, L.status);
  int32_t* topk_idx = at<int32_t>(ctx, L.topk_idx);
  float* gates = at<float>(ctx, L.gates);
  int32_t* offsets = at<int32_t>(ctx, L.offsets);
  int32_t* tile_off = at<int32_t>(ctx, L.tile_off);
  int32_t* row_of = at<int32_t>(ctx, L.row_of);
  int32_t* src_of = at<int32_t>(ctx, L.src_of);
  float* hu = at<float>(ctx, L.hu);
  float* o = at<float>(ws, L.expert_out);
  float* logits = at<float>(ws, L.logits);
  int32_t* blk_off = at<int32_t>(ws, L.mx_blk_off);
  void* xq = at<char>(ws, L.mx_xq);
  void* xsf = at<char>(ws, L.mx_xsf);
  void* aq = at<char>(ws, L.mx_aq);
  void* asf = at<char>(ws, L.mx_asf);
  const int RP = (int)mok::mx_rows_padded_bound(R, E), G = (int)mok::mx_row_groups(R, E);

  MOK_CUDA(cudaMemsetAsync(status, 0, mok::STATUS_BYTES, st));
  MOK_LAUNCH("router_gemm", st, mok::launch_router_gemm(x, w_router, T, H, E, logits, status, n_sm, st));
  MOK_LAUNCH("topk", st, mok::launch_topk(logits, router_bias, given_topk, T, E, k, d->router, d->renorm,
                                          d->route_scale, topk_idx, gates, at<float>(ctx, L.scores), status, st));
  MOK_LAUNCH("schedule", st, mok::launch_schedule_multi(topk_idx, gates, R, E, at<int32_t>(ctx, L.counts), offsets,
                                                        row_of, src_of, tile_off, at<float>(ctx, L.gate_row),
                                                        at<int32_t>(ws, L.sched), status, st));
  // each expert's rows padded to 32 in the E4M3 row space of the FP8 GEMMs
  MOK_LAUNCH("mx_block_offsets", st, mok::launch_mx_block_offsets(offsets, E, blk_off, st));
  // pull dispatch with the MXFP8 quantisation of each row along H (E4M3 bytes + scale blocks)
  MOK_LAUNCH("gather_x_mx", st, mok::launch_gather_rows_mxf8(x, src_of, topk_idx, offsets, blk_off, k, R, H, E, xq,
                                                             xsf, st));
  // GEMM1 on the FP8 tensor path, SwiGLU, a quantised along I (E4M3 bytes + scale blocks)
  MOK_LAUNCH("gemm1_swiglu_mx", st, mok::launch_gemm1_swiglu_mxf8(xq, xsf, w13_q, w13_scale, RP, G, R, H, I, E, offsets,
                                                                  blk_off, hu, aq, asf, status, n_sm, st));
  MOK_LAUNCH("gemm2_mx", st, mok::launch_gemm2_mxf8(aq, asf, w2_q, w2_scale, RP, G, R, H, I, E, offsets, blk_off, o,
                                                    status, n_sm, st));
  MOK_LAUNCH("combine", st, mok::launch_combine(o, gates, row_of, T, k, H, nullptr, nullptr, nullptr, E, 0, y, n_sm, st));
  return MOK_OK;
}

mok_status mok_moe_backward(const mok_layer_desc* d, const void* dy, const void* x, const void* w_router,
                            const void* w13, const void* w2, const void* ctx, size_t ctx_bytes, void* dx,
                            float* dw_router, void* dw13, void* dw2, float* dgates, void* ws, size_t ws_bytes,
                            void* stream) {
  mok_status s = check_desc(d);
  if (s != MOK_OK) return s;
  if (d->precision != MOK_BF16) return MOK_ERR_UNSUPPORTED;
  if (!dy || !x || !w_router || !w13 || !w2 || !ctx || !dx || !dw_router || !dw13 || !dw2 || !ws)
    return MOK_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(w_router) || !aligned16(w13) || !aligned16(w2) ||
      !aligned16(ctx) || !aligned16(dx) || !aligned16(dw_router) || !aligned16(dw13) || !aligned16(dw2) ||
      !aligned16(ws))
    return MOK_ERR_INVALID_ARG;
  mok_layout L;
  s = fill_layout(d, &L);
  if (s != MOK_OK) return s;
  if ((int64_t)ctx_bytes < L.ctx_bytes || (int64_t)ws_bytes < L.ws_bytes) return MOK_ERR_WORKSPACE_TOO_SMALL;
  const int n_sm = sm_count();
  if (n_sm <= 0) return MOK_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = d->T, H = d->H, I = d->I, E = d->E, k = d->k, R = T * k;
  int* status = at<int>(ws, L.status);
  // the work counters of this call start at zero (the status word keeps what the forward left)
  MOK_CUDA(cudaMemsetAsync(status + mok::STATUS_COUNTERS, 0, mok::STATUS_BYTES - 4 * mok::STATUS_COUNTERS, st));
  if (d->ring_bytes > 0) {
    // Ring backward: the ring forward left the dispatched rows of its last `slots` minibatches in
    // the ring, at their own rows of the dispatched-row region of ws; replay (gather again) only
    // the minibatches it overwrote, in front of them.  If ws is not the one that forward filled
    // (its stamp differs from ctx's), every row is replayed; the rows are the same either way.
    RingGeom rg;
    s = ring_geometry(d, &rg);
    if (s != MOK_OK) return s;
    const int32_t* cnt = at<int32_t>(ws, L.mb_counters);
    MOK_LAUNCH("gather_x_replay", st,
               mok::launch_ring_replay(
                   x, at<int32_t>(ctx, L.src_of), k, R, H, at<char>(ws, L.ring), (rg.n_mb - rg.slots) * rg.m,
                   reinterpret_cast<const unsigned long long*>(reinterpret_cast<const char*>(cnt) +
                                                               ring_stamp_offset(rg.n_mb)),
                   at<unsigned long long>(ctx, L.ring_stamp), (unsigned long long)reinterpret_cast<uintptr_t>(ctx), st));
  }
  const int32_t* topk_idx = at<int32_t>(ctx, L.topk_idx);
  const float* gates = at<float>(ctx, L.gates);
  const float* scores = at<float>(ctx, L.scores);
  const int32_t* offsets = at<int32_t>(ctx, L.offsets);
  const int32_t* tile_off = at<int32_t>(ctx, L.tile_off);
  const int32_t* row_of = at<int32_t>(ctx, L.row_of);
  const int32_t* src_of = at<int32_t>(ctx, L.src_of);
  const float* gate_row = at<float>(ctx, L.gate_row);
  const void* x_g = d->ring_bytes > 0 ? static_cast<const void*>(at<char>(ws, L.ring))
                                      : static_cast<const void*>(at<char>(ctx, L.x_g));
  const float* hu = at<float>(ctx, L.hu);
  void* dy_g = at<char>(ws, L.dy_g);
  void* dhu = at<char>(ws, L.dhu);
  void* dhu_lo = at<char>(ws, L.dhu_lo);
  void* gact = at<char>(ws, L.gact);
  void* gact_lo = at<char>(ws, L.gact_lo);
  float* dx_g = at<float>(ws, L.dx_g);
  float* dg_part = at<float>(ws, L.dg_part);
  float* dl = at<float>(ws, L.dlogits);
  const int wgrad_f32 = (d->flags & MOK_FLAG_WGRAD_BF16) ? 0 : 1;

  // 1. reverse combine: pull the upstream gradient rows into expert order
  MOK_LAUNCH("gather_dy", st, mok::launch_gather_rows(dy, src_of, k, R, H, dy_g, n_sm, st));
  // 2. dA' = dY_g W2[e]; epilogue: SwiGLU backward, g * a, and per-tile <dA', a>
  MOK_LAUNCH("dgrad_swiglu", st, mok::launch_dgrad_swiglu(dy_g, w2, R, H, I, E, offsets, tile_off, hu, gate_row, dhu,
                                                          dhu_lo, gact, gact_lo, dg_part, status, n_sm, st));
  // 3. dX_g = [dh | du] W13[e]
  MOK_LAUNCH("dgrad_x", st, mok::launch_dgrad_x(dhu, dhu_lo, w13, R, H, I, E, offsets, tile_off, dx_g, status, n_sm,
                                                gemm_variant(d, DGRAD_X), st));
  // 4. dW2[e] = (g a)^T dY_g stored as [H][I]; 5. dW13[e] = x_g^T [dh | du] stored as [2I][H];
  //    both reduced over the expert's rows, the contiguous output dimension on the TMEM lanes
  MOK_LAUNCH("wgrad_w2", st, mok::launch_wgrad(gact, gact_lo, I, dy_g, nullptr, H, R, E, offsets, dw2, wgrad_f32,
                                               status, status + mok::STATUS_COUNTERS + mok::CNT_WGRAD_W2,
                                               wgrad_pairs(d), n_sm, st));
  MOK_LAUNCH("wgrad_w13", st, mok::launch_wgrad(x_g, nullptr, H, dhu, dhu_lo, 2 * I, R, E, offsets, dw13, wgrad_f32,
                                                status, status + mok::STATUS_COUNTERS + mok::CNT_WGRAD_W13,
                                                wgrad_pairs(d), n_sm, st));
  // 6. gate and router-logit gradients, 7. router weight gradient
  MOK_LAUNCH("router_dlogits", st, mok::launch_router_dlogits(dg_part, (I + 255) / 256, row_of, topk_idx, gates, scores, T, E, k, d->router,
                                      d->renorm, d->route_scale, dgates, dl, st));
  MOK_LAUNCH("router_wgrad", st, mok::launch_router_wgrad(dl, x, offsets, src_of, T, H, E, k, d->router == MOK_ROUTER_SIGMOID ? 1 : 0,
                                    dw_router, st));
  // 8. reverse dispatch: dX[t] = sum_j dX_g[row_of[t,j]] + dl[t] W_r
  MOK_LAUNCH("combine_dx", st, mok::launch_combine(dx_g, nullptr, row_of, T, k, H, dl, w_router, topk_idx, E,
                               d->router == MOK_ROUTER_SOFTMAX ? 1 : 0, dx, n_sm, st));
  return MOK_OK;
}

mok_status mok_read_status(void* ws, size_t ws_bytes, void* stream, int32_t* device_status) {
  if (!ws || !device_status || ws_bytes < 16) return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status word is the first tensor of ws
  MOK_CUDA(cudaMemcpyAsync(device_status, ws, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  MOK_CUDA(cudaStreamSynchronize(st));
  MOK_CUDA(cudaMemsetAsync(ws, 0, 16, st));
  MOK_CUDA(cudaStreamSynchronize(st));
  return MOK_OK;
}

mok_status mok_test_bounded_wait(void* ws, size_t ws_bytes, int32_t limit_ms, void* stream) {
  if (!ws || ws_bytes < 16 || limit_ms < 1 || limit_ms > 10000) return MOK_ERR_INVALID_ARG;
  MOK_LAUNCH("test_wait", static_cast<cudaStream_t>(stream), mok::launch_test_wait(static_cast<int*>(ws), (long long)limit_ms * 1000000LL,
                                 static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

mok_status mok_trace_start(int32_t max_launches) {
  if (max_launches < 1 || max_launches > (1 << 20)) return MOK_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_trace.mu);
  if (g_trace.on) return MOK_ERR_INVALID_ARG;
  g_trace.recs = new (std::nothrow) TraceRec[max_launches];
  if (!g_trace.recs) return MOK_ERR_INVALID_ARG;
  for (int i = 0; i < max_launches; ++i) {
    if (cudaEventCreate(&g_trace.recs[i].start) != cudaSuccess ||
        cudaEventCreate(&g_trace.recs[i].stop) != cudaSuccess) {
      for (int j = 0; j < i; ++j) {
        cudaEventDestroy(g_trace.recs[j].start);
        cudaEventDestroy(g_trace.recs[j].stop);
      }
      delete[] g_trace.recs;
      g_trace.recs = nullptr;
      return MOK_ERR_CUDA;
    }
  }
  g_trace.cap = max_launches;
  g_trace.used = 0;
  g_trace.on = true;
  return MOK_OK;
}

mok_status mok_trace_stop(mok_trace_entry* out, int32_t cap, int32_t* n_out) {
  std::lock_guard<std::mutex> lock(g_trace.mu);
  if (!g_trace.on) return MOK_ERR_INVALID_ARG;
  g_trace.on = false;
  mok_status st = MOK_OK;
  int n = 0;
  for (int i = 0; i < g_trace.used; ++i) {
    TraceRec& r = g_trace.recs[i];
    float ms = 0.0f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
      st = MOK_ERR_CUDA;
      continue;
    }
    int slot = -1;
    for (int j = 0; j < n; ++j)
      if (std::strncmp(out[j].name, r.name, sizeof(out[j].name)) == 0) slot = j;
    if (slot < 0) {
      if (out == nullptr || n >= cap) continue;
      slot = n++;
      std::memset(out[slot].name, 0, sizeof(out[slot].name));
      std::strncpy(out[slot].name, r.name, sizeof(out[slot].name) - 1);
      out[slot].launches = 0;
      out[slot].total_ms = 0.0f;
    }
    out[slot].launches += 1;
    out[slot].total_ms += ms;
  }
  for (int i = 0; i < g_trace.cap; ++i) {
    cudaEventDestroy(g_trace.recs[i].start);
    cudaEventDestroy(g_trace.recs[i].stop);
  }
  delete[] g_trace.recs;
  g_trace.recs = nullptr;
  g_trace.cap = g_trace.used = 0;
  if (n_out) *n_out = n;
  return st;
}

}  // extern "C"
