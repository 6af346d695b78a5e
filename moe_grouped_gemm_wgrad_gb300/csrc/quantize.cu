// MXFP8 quantization of a wgrad operand: bf16 [M, C] (token-major) -> e4m3
// [C, Mcap] (token-contiguous, per-expert 128-padded) + e8m0 scale atoms.
//
// HBM-bound transpose-quantize.  One work unit is 128 padded tokens x 128
// features: it reads up to 32 KB of bf16 with 16-byte coalesced loads, finds
// each (feature, 32-token block) maximum, scales by an exact power of two,
// converts with the hardware's round-to-nearest-even saturating e4m3 convert,
// and writes a 16 KB e4m3 tile (full 128-byte rows) plus one 512-byte scale
// atom.  A persistent grid walks the units.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace mgw {
namespace {

constexpr int kThreads = 256;
constexpr int kIn = 128 * 128 * 2;   // bf16 input tile [token][feature]
constexpr int kOutPitch = 144;       // bytes per feature row of the e4m3 tile (128 + 16 pad)
constexpr int kOut = 128 * kOutPitch;
constexpr int kSf = 512;

__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

__global__ void __launch_bounds__(kThreads) mxfp8_quantize_kernel(
    const uint16_t* __restrict__ src, int M, int C, const int32_t* __restrict__ expert_off, int E,
    uint8_t* __restrict__ q, uint8_t* __restrict__ sc, long long Mcap, int* status) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* s_in = reinterpret_cast<uint16_t*>(smem);
  uint8_t* s_out = smem + kIn;
  uint8_t* s_sf = smem + kIn + kOut;
  int* s_off = reinterpret_cast<int*>(smem + kIn + kOut + kSf);
  int* s_pad = s_off + (E + 1);
  int* s_flag = s_pad + (E + 1);
  if (!load_offsets(expert_off, E, M, s_off, s_pad, s_flag, status)) return;

  const int tid = threadIdx.x;
  const int col_tiles = C / 128;
  const long long units = (Mcap / 128) * col_tiles;
  const int used_chunks = s_pad[E] / 128;

  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const int ch = static_cast<int>(u / col_tiles);
    const int ct = static_cast<int>(u % col_tiles);
    // Expert of this 128-token chunk of the padded axis: the largest e with
    // P[e] <= 128*ch (always a non-empty expert when the chunk is in use).
    int valid = 0, row0 = 0;
    if (ch < used_chunks) {
      const int t0 = ch * 128;
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pad[mid] <= t0)
          lo = mid;
        else
          hi = mid - 1;
      }
      const int tin = t0 - s_pad[lo];
      const int cnt = s_off[lo + 1] - s_off[lo];
      valid = min(128, cnt - tin);
      row0 = s_off[lo] + tin;
    }
    // Load the bf16 tile: 128 tokens x 16 x 16 B; tokens past the expert's end are zero.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = tid + i * kThreads;
      const int r = idx >> 4, c16 = idx & 15;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < valid)
        v = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(row0 + r) * C +
                                                 ct * 128 + c16 * 8));
      *reinterpret_cast<uint4*>(s_in + r * 128 + c16 * 8) = v;
    }
    __syncthreads();
    // Quantize: thread -> feature c, two 32-token blocks.
    const int c = tid & 127;
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      const int kb = (tid >> 7) * 2 + bb;
      uint32_t h[32];
      uint32_t amax = 0;
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        h[t] = s_in[(kb * 32 + t) * 128 + c];
        amax = max(amax, h[t] & 0x7FFFu);  // |bf16| orders like its bits (finite values)
      }
      // floor(log2 amax) = exponent field - 127 for normal bf16; the scale byte is
      // that minus 8 plus the bias 127, clamped at 0 (which also covers amax == 0
      // and every subnormal amax).
      const int ef = static_cast<int>(amax >> 7);
      const int byte = ef > 8 ? ef - 8 : 0;
      const float inv = __uint_as_float(static_cast<uint32_t>(254 - byte) << 23);  // 2^(127-byte)
      uint32_t pk[8];
#pragma unroll
      for (int t = 0; t < 32; t += 4)
        pk[t / 4] = cvt_e4m3x4(bf16_bits_to_float(h[t]) * inv, bf16_bits_to_float(h[t + 1]) * inv,
                               bf16_bits_to_float(h[t + 2]) * inv, bf16_bits_to_float(h[t + 3]) * inv);
      uint4* dst = reinterpret_cast<uint4*>(s_out + c * kOutPitch + kb * 32);
      dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      s_sf[(c & 31) * 16 + ((c >> 5) & 3) * 4 + kb] = static_cast<uint8_t>(byte);
    }
    __syncthreads();
    // Store: 128 feature rows x 128 B (8 threads per row), then the 512-byte atom.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (tid >> 3) + i * 32, c16 = tid & 7;
      const uint4 v = *reinterpret_cast<const uint4*>(s_out + r * kOutPitch + c16 * 16);
      *reinterpret_cast<uint4*>(q + static_cast<size_t>(ct * 128 + r) * static_cast<size_t>(Mcap) +
                                static_cast<size_t>(ch) * 128 + c16 * 16) = v;
    }
    if (tid < 32) {
      const uint4 v = *reinterpret_cast<const uint4*>(s_sf + tid * 16);
      *reinterpret_cast<uint4*>(sc + (static_cast<size_t>(ch) * col_tiles + ct) * kSf + tid * 16) = v;
    }
    __syncthreads();
  }
}

}  // namespace

size_t quantize_smem_bytes(int E) {
  return static_cast<size_t>(kIn + kOut + kSf) + sizeof(int) * (2 * (E + 1) + 1);
}

cudaError_t launch_mxfp8_quantize(const void* src, int M, int C, const int32_t* expert_off, int E,
                                  void* q, void* sc, long long Mcap, int* status, int num_sms,
                                  cudaStream_t stream) {
  const size_t smem = quantize_smem_bytes(E);
  static thread_local int attr_set_device = -1;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (attr_set_device != dev) {
    err = cudaFuncSetAttribute(mxfp8_quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(quantize_smem_bytes(kMaxExperts)));
    if (err != cudaSuccess) return err;
    attr_set_device = dev;
  }
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mxfp8_quantize_kernel, kThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const long long units = (Mcap / 128) * (C / 128);
  long long grid = static_cast<long long>(num_sms) * per_sm;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  mxfp8_quantize_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(
      static_cast<const uint16_t*>(src), M, C, expert_off, E, static_cast<uint8_t*>(q),
      static_cast<uint8_t*>(sc), Mcap, status);
  return cudaGetLastError();
}

}  // namespace mgw
