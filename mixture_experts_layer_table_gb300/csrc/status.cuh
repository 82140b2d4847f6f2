// Device-side status word: the first error a kernel meets is recorded here (code, site)
// and read back by the host after a stream synchronisation; kernels never trap.
#pragma once
#include <cstdint>

namespace mok {

// Codes match mok_status in include/mok.h.
constexpr int MOK_DEV_OK = 0;
constexpr int MOK_DEV_TIMEOUT = 5;
constexpr int MOK_DEV_INVALID_ROUTING = 6;

// Sites, for the second status word (which wait or check fired).
enum StatusSite : int {
  SITE_NONE = 0,
  SITE_GEMM_PRODUCER_EMPTY = 1,
  SITE_GEMM_MMA_FULL = 2,
  SITE_GEMM_MMA_TMEM_EMPTY = 3,
  SITE_GEMM_EPI_TMEM_FULL = 4,
  SITE_GEMM_DRAIN = 5,
  SITE_TOPK_INDEX = 10,
  SITE_SCHEDULE_INDEX = 11,
  SITE_RING_WAIT = 20,
  SITE_TEST_WAIT = 30,
};

// status[0] = code of the first error, status[1] = its site.
__device__ __forceinline__ void report_status(int* status, int code, int site) {
  if (status == nullptr) return;
  if (atomicCAS(&status[0], 0, code) == 0) {
    atomicExch(&status[1], site);
  }
}

}  // namespace mok
