// Router + schedule table without any caller-provided workspace.
//
// mok_schedule needs a workspace `ws` for its scratch (the device status word and, when the
// router runs, the fp32 router logits).  Some callers cannot allocate device memory at the
// point where they route tokens: code running under an allocator that forbids new
// allocations (a captured or replayed step whose memory plan is fixed), an inference
// runtime that hands out only its own pre-sized buffers, or a C caller without any CUDA
// allocator of its own.  mok_schedule_noalloc serves them: its scratch is a fixed array
// compiled into the library, so the caller passes only inputs and outputs.
//
// The array lives in every GPU's memory that loads the library, until the process exits,
// and every call on a device shares it.  Calls whose kernels overlap on the GPU (two
// streams, or two host threads) race on it; callers must order them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernels.cuh"
#include "mok.h"

namespace {

constexpr size_t kStatusBytes = 256;  // status word, padded so the logits start 256-aligned
constexpr size_t kScratchBytes = kStatusBytes + size_t(MOK_NOALLOC_MAX_LOGITS) * sizeof(float);
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the symbol, never a
// device address: the address is looked up per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
CUcontext g_scratch_ctx[kMaxDevices] = {nullptr};
int g_sm_count[kMaxDevices] = {0};

// The driver's cuCtxGetCurrent, found through the runtime (the library does not link libcuda).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Looks up (once per device and context, with that device current) the device address of the
// scratch array and the SM count.  The address is kept together with the context it was looked
// up in: after a context is destroyed and created again (cudaDeviceReset) the module may load at
// another address, so a new context means a new lookup.  Returns false when the lookup fails.
bool setup_current_device(void** scratch, int* n_sm) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  // make the device's primary context current (cudaSetDevice initialises it) before asking which it is
  if (cudaSetDevice(dev) != cudaSuccess) return false;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  CUcontext ctx = nullptr;
  if (get_ctx == nullptr || get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return false;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return false;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
    g_sm_count[dev] = n;
  }
  *scratch = g_scratch_ptr[dev];
  *n_sm = g_sm_count[dev];
  return true;
}

}  // namespace

extern "C" mok_status mok_schedule_noalloc(const mok_layer_desc* d, const void* x, const void* w_router,
                                           const float* router_bias, const int32_t* given_topk,
                                           int32_t* topk_idx, float* gates, int32_t* counts, int32_t* offsets,
                                           int32_t* row_of, int32_t* src_of, int32_t* device_status,
                                           void* stream) {
  mok_layout L;
  const mok_status s = mok_get_layout(d, &L);  // validates the descriptor
  if (s != MOK_OK) return s;
  if (!topk_idx || !counts || !offsets || !row_of || !src_of) return MOK_ERR_INVALID_ARG;
  const bool have_router = x != nullptr && w_router != nullptr;
  if (!have_router && (given_topk == nullptr || gates != nullptr)) return MOK_ERR_INVALID_ARG;
  if (have_router && ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w_router) & 15u)))
    return MOK_ERR_INVALID_ARG;
  // the router logits of this call must fit the fixed scratch
  if (have_router && int64_t(d->T) * d->E > int64_t(MOK_NOALLOC_MAX_LOGITS)) return MOK_ERR_WORKSPACE_TOO_SMALL;

  void* scratch = nullptr;
  int n_sm = 0;
  if (!setup_current_device(&scratch, &n_sm)) return MOK_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(scratch);
  float* logits = reinterpret_cast<float*>(static_cast<char*>(scratch) + kStatusBytes);

  // the status word keeps the previous call's contents: clear it first
  if (cudaMemsetAsync(status, 0, 16, st) != cudaSuccess) return MOK_ERR_CUDA;
  if (have_router &&
      mok::launch_router_gemm(x, w_router, d->T, d->H, d->E, logits, status, n_sm, st) != cudaSuccess)
    return MOK_ERR_CUDA;
  if (mok::launch_topk(have_router ? logits : nullptr, router_bias, given_topk, d->T, d->E, d->k, d->router,
                       d->renorm, d->route_scale, topk_idx, gates, nullptr, status, st) != cudaSuccess)
    return MOK_ERR_CUDA;
  if (mok::launch_schedule(topk_idx, nullptr, d->T * d->k, d->E, counts, offsets, row_of, src_of, nullptr, nullptr,
                           status, st) != cudaSuccess)
    return MOK_ERR_CUDA;
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, status, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MOK_ERR_CUDA;
  return MOK_OK;
}
