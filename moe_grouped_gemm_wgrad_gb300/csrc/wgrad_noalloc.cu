// The load-balanced grouped wgrad on a library-owned workspace: a file-scope device array
// (zero-filled when the module loads, kept zero between calls by the kernel itself), so the
// call allocates nothing and needs no workspace argument.  Its address is looked up once per
// device with cudaGetSymbolAddress.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace mgw {
namespace {

// Header (item and CTA counters), 128 tile counters padded to 256 bytes, 128 fp32 partial
// tiles of 128 x 256 (16 MB).
constexpr int kNoAllocSlots = 128;
constexpr size_t kNoAllocBytes =
    kWsHeaderBytes + ((4 * static_cast<size_t>(kNoAllocSlots) + 255) & ~size_t(255)) +
    static_cast<size_t>(kNoAllocSlots) * 128 * 256 * 4;

static __device__ __align__(256) uint8_t g_wgrad_workspace[kNoAllocBytes];

}  // namespace

cudaError_t noalloc_wgrad_workspace(void** ptr, size_t* bytes) {
  static std::mutex mu;
  static void* cached[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == nullptr) {
    err = cudaGetSymbolAddress(&cached[dev], g_wgrad_workspace);
    if (err != cudaSuccess) return err;
  }
  *ptr = cached[dev];
  *bytes = kNoAllocBytes;
  return cudaSuccess;
}

}  // namespace mgw
