// Diagnostics of the diagnostic library libmgw_diag.so (every translation unit compiled with
// MGW_DIAG; libmgw.so has none of this):
//   * a work-item timeline: per CTA and work item, the globaltimer when the item's epilogue
//     began waiting for its accumulator and when the item's results were stored, with the
//     SM that ran it, appended to a per-kernel device buffer that the host reads back
//     (mgw_diag_timeline in the C ABI);
//   * device bounds checks on the global addresses the kernels compute for their stores and
//     TMA loads: a store outside its output is skipped and a load outside its tensor is
//     reported (TMA fills it with zeros), both by OR-ing kDevBounds into the status word.
// In libmgw.so MGW_DIAG_CHECK is `true` and the timeline calls compile to nothing.
#pragma once
#include <cstdint>

#include "kernels.h"

namespace mgw {

constexpr int kDevBounds = 8;  // a computed global address outside its tensor (diag build)

#ifdef MGW_DIAG
__device__ __forceinline__ bool diag_check(bool ok, int* status) {
  if (!ok && status != nullptr) atomicOr(status, kDevBounds);
  return ok;
}
#define MGW_DIAG_CHECK(cond, status) (::mgw::diag_check((cond), (status)))

__device__ __forceinline__ uint64_t diag_now() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t diag_smid() {
  uint32_t s;
  asm volatile("mov.u32 %0, %smid;" : "=r"(s));
  return s;
}

// One timeline buffer per kernel family (per translation unit); the host side of each is
// declared in kernels.h.
#define MGW_DIAG_TIMELINE_DEFINE(family, kernel_id)                                           \
  static __device__ DiagRecord g_diag_tl_##family[kDiagTimelineCap];                          \
  static __device__ unsigned int g_diag_tl_n_##family;                                         \
  __device__ __forceinline__ void diag_item_##family(long long item, uint64_t t0, uint64_t t1) { \
    const unsigned int i = atomicAdd(&g_diag_tl_n_##family, 1u);                               \
    if (i < static_cast<unsigned int>(kDiagTimelineCap)) {                                    \
      DiagRecord r;                                                                            \
      r.kernel = (kernel_id);                                                                  \
      r.sm = diag_smid();                                                                      \
      r.cta = blockIdx.x;                                                                      \
      r.pad = 0;                                                                               \
      r.item = item;                                                                           \
      r.t_wait = t0;                                                                           \
      r.t_done = t1;                                                                           \
      g_diag_tl_##family[i] = r;                                                               \
    }                                                                                          \
  }                                                                                            \
  cudaError_t diag_timeline_read_##family(DiagRecord* host, int cap, int* count) {            \
    unsigned int n = 0;                                                                        \
    cudaError_t err = cudaMemcpyFromSymbol(&n, g_diag_tl_n_##family, sizeof(n));               \
    if (err != cudaSuccess) return err;                                                        \
    const int avail = static_cast<int>(n < static_cast<unsigned int>(kDiagTimelineCap)        \
                                           ? n : static_cast<unsigned int>(kDiagTimelineCap)); \
    const int m = avail < cap ? avail : cap;                                                   \
    *count = static_cast<int>(n);                                                              \
    if (m > 0)                                                                                 \
      err = cudaMemcpyFromSymbol(host, g_diag_tl_##family, sizeof(DiagRecord) * m);           \
    return err;                                                                                \
  }                                                                                            \
  cudaError_t diag_timeline_reset_##family() {                                                 \
    const unsigned int zero = 0;                                                               \
    return cudaMemcpyToSymbol(g_diag_tl_n_##family, &zero, sizeof(zero));                      \
  }
#define MGW_DIAG_ITEM(family, item, t0, t1) diag_item_##family((item), (t0), (t1))
#define MGW_DIAG_NOW() ::mgw::diag_now()
#else
#define MGW_DIAG_CHECK(cond, status) (true)
#define MGW_DIAG_TIMELINE_DEFINE(family, kernel_id)
#define MGW_DIAG_ITEM(family, item, t0, t1) ((void)0)
#define MGW_DIAG_NOW() (uint64_t{0})
#endif

}  // namespace mgw
