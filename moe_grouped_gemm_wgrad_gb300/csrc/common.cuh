// Shared device helpers: reading and checking the expert offsets, and the
// padded token layout of the quantized operands.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace mgw {

// Loads expert_off[0..E] into shared memory, checks 0 = off[0] <= ... <= off[E] = total,
// and computes the 128-padded segment starts P[0..E] (P[e+1] = P[e] + ceil128(count_e)).
// Must be called by all threads of the block; returns false (uniformly) when the
// offsets are invalid, after reporting kDevBadOffsets once per block.
__device__ __forceinline__ bool load_offsets(const int32_t* __restrict__ expert_off, int E,
                                             int total, int* s_off, int* s_pad, int* s_flag,
                                             int* status) {
  if (threadIdx.x == 0) *s_flag = 0;
  __syncthreads();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = expert_off[i];
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    if (s_off[i + 1] < s_off[i]) *s_flag = 1;
  if (threadIdx.x == 0 && (s_off[0] != 0 || s_off[E] != total)) *s_flag = 1;
  __syncthreads();
  const bool bad = *s_flag != 0;
  if (bad) {
    if (threadIdx.x == 0 && status != nullptr) atomicOr(status, kDevBadOffsets);
    return false;
  }
  // Exclusive scan of ceil128(counts) by warp 0, 32 experts per step.
  if (threadIdx.x < 32) {
    const uint32_t lane = threadIdx.x;
    int carry = 0;
    if (lane == 0) s_pad[0] = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + static_cast<int>(lane);
      int v = (e < E) ? ((s_off[e + 1] - s_off[e] + 127) & ~127) : 0;
      // inclusive scan within the warp
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= static_cast<uint32_t>(d)) v += y;
      }
      if (e < E) s_pad[e + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  return true;
}

}  // namespace mgw
