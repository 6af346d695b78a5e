// The load-balanced grouped wgrad on a library-owned workspace: a file-scope device array
// (zero-filled when the module loads), so the call allocates nothing and needs no workspace
// argument.  Its address is looked up with cudaGetSymbolAddress once per CUDA context (keyed
// on the context's unique id, so a context re-created after cudaDeviceReset looks it up
// again instead of reusing a stale address).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace mgw {
namespace {

// Header (item and CTA counters), 128 tile counters padded to 256 bytes, 128 fp32 partial
// tiles of 128 x 256 (16 MB).
constexpr int kNoAllocSlots = 128;
constexpr size_t kNoAllocCounterBytes =
    kWsHeaderBytes + ((4 * static_cast<size_t>(kNoAllocSlots) + 255) & ~size_t(255));
constexpr size_t kNoAllocBytes =
    kNoAllocCounterBytes + static_cast<size_t>(kNoAllocSlots) * 128 * 256 * 4;

static __device__ __align__(256) uint8_t g_wgrad_workspace[kNoAllocBytes];

struct Lookup {
  uint64_t ctx = 0;
  void* ptr = nullptr;
};

}  // namespace

cudaError_t noalloc_wgrad_workspace(void** ptr, size_t* bytes, size_t* counter_bytes) {
  static std::mutex mu;
  static Lookup cached[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  const uint64_t ctx = current_context_id();
  if (ctx == 0 || cached[dev].ctx != ctx) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_wgrad_workspace);
    if (err != cudaSuccess) return err;
    // The lookup made the device's context current if none was; key the cache on it.
    cached[dev].ctx = current_context_id();
    cached[dev].ptr = p;
  }
  *ptr = cached[dev].ptr;
  *bytes = kNoAllocBytes;
  *counter_bytes = kNoAllocCounterBytes;
  return cudaSuccess;
}

}  // namespace mgw
