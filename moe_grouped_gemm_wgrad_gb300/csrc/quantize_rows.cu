// Row-wise MXFP8 quantization for the forward and data-gradient GEMMs: bf16 [rows, C]
// -> e4m3 [Mcap, C] (row-major, no transpose) + e8m0 scale atoms, one scale per 32
// consecutive elements of a row.  Routed row r of expert e lands on padded row
// P[e] + (r - off[e]), so every expert's rows start on a 128-row boundary and the
// GEMM's 128-row tiles never mix experts; padding rows are zero.
//
// HBM-bound streaming.  One warp quantizes one padded row at a time: lane l owns
// 8 consecutive elements of each 256-element segment (one 16-byte load, coalesced
// 512 bytes per warp instruction), the block maximum is reduced over the 4 lanes of a
// 32-element block with two shuffles, and the 8 e4m3 bytes leave as one 8-byte store
// (256 bytes per warp instruction).  Up to eight segments' loads are in flight per
// warp before any is used.  The four scale bytes of a 128-element chunk form one
// 32-bit word of the chunk's 512-byte atom (row p % 128 = r0 + 32 r1 at byte
// 16 r0 + 4 r1 + block), written by the chunk's first lane.
//
// A gathered source (row_index != nullptr) reads routed row r from row row_index[r] of
// the unpermuted token matrix; indices outside [0, src_rows) give zero rows and set
// kDevBadIndex.
#include <cuda_bf16.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "mx.cuh"

namespace mgw {
namespace {

constexpr int kRThreads = 256;
constexpr int kRWarps = kRThreads / 32;
constexpr int kSegs = 8;  // segments (256 elements each) loaded ahead per warp

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t abs_max_bf16x2(uint32_t m, uint32_t w) {
  return max(m, max(w & 0x7FFFu, (w >> 16) & 0x7FFFu));  // |bf16| orders like its bits
}

__global__ void __launch_bounds__(kRThreads, 4) mxfp8_quantize_rows_kernel(
    const uint16_t* __restrict__ src, int src_rows, const int32_t* __restrict__ row_index, int M,
    int C, const int32_t* __restrict__ expert_off, int E, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sc, long long Mcap, int rule, int* status) {
  extern __shared__ int s_tab[];
  int* s_off = s_tab;
  int* s_pad = s_off + (E + 1);
  int* s_flag = s_pad + (E + 1);
  if (!load_offsets(expert_off, E, M, s_off, s_pad, s_flag, status)) return;

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const uint32_t lane = lane_id();
  const long long used = s_pad[E];
  const int nseg = (C + 255) / 256;
  const long long row_tiles = Mcap / 128;
  const long long step = static_cast<long long>(gridDim.x) * kRWarps;

  for (long long p = static_cast<long long>(blockIdx.x) * kRWarps + warp; p < Mcap; p += step) {
    // Source row of padded row p, or -1 for a padding row.
    long long srow = -1;
    if (p < used) {
      int lo = 0, hi = E - 1;  // the largest e with P[e] <= p: a non-empty expert
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pad[mid] <= p)
          lo = mid;
        else
          hi = mid - 1;
      }
      const long long i = p - s_pad[lo];
      if (i < s_off[lo + 1] - s_off[lo]) {
        const long long r = s_off[lo] + i;
        srow = r;
        if (row_index != nullptr) {
          const int idx = row_index[r];
          if (idx < 0 || idx >= src_rows) {
            if (lane == 0 && status != nullptr) atomicOr(status, kDevBadIndex);
            srow = -1;
          } else {
            srow = idx;
          }
        }
      }
    }
    const uint16_t* srcrow = src + (srow < 0 ? 0 : srow) * static_cast<long long>(C);
    uint8_t* qrow = q + p * static_cast<long long>(C);
    const long long atom_row = p / 128;
    const uint32_t in_atom = 16u * static_cast<uint32_t>(p & 31) + 4u * static_cast<uint32_t>((p & 127) >> 5);
    for (int s0 = 0; s0 < nseg; s0 += kSegs) {
      uint4 v[kSegs];
#pragma unroll
      for (int i = 0; i < kSegs; ++i) {
        const int col = (s0 + i) * 256 + 8 * static_cast<int>(lane);
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (srow >= 0 && col < C) v[i] = ld_stream_v4(srcrow + col);
      }
#pragma unroll
      for (int i = 0; i < kSegs; ++i) {
        const int seg = s0 + i;
        if (seg >= nseg) break;  // uniform over the warp
        const int col = seg * 256 + 8 * static_cast<int>(lane);
        uint32_t m = 0;
        m = abs_max_bf16x2(m, v[i].x);
        m = abs_max_bf16x2(m, v[i].y);
        m = abs_max_bf16x2(m, v[i].z);
        m = abs_max_bf16x2(m, v[i].w);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        float inv;
        int byte = scale_byte(m, rule, &inv);
        if (srow < 0) byte = 0;  // padding row (its values are zero: inv is irrelevant)
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f[2 * j] = __uint_as_float(w[j] << 16) * inv;
          f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u) * inv;
        }
        const uint2 out = make_uint2(cvt_e4m3x4(f[0], f[1], f[2], f[3]),
                                     cvt_e4m3x4(f[4], f[5], f[6], f[7]));
        if (col < C) *reinterpret_cast<uint2*>(qrow + col) = out;
        // Lanes 0-15 hold chunk 2*seg, lanes 16-31 chunk 2*seg+1; block kb of a chunk is
        // lanes base + 4kb .. base + 4kb + 3.
        const int base = static_cast<int>(lane & 16u);
        const uint32_t b = static_cast<uint32_t>(byte);
        const uint32_t word = __shfl_sync(0xffffffffu, b, base) |
                              (__shfl_sync(0xffffffffu, b, base + 4) << 8) |
                              (__shfl_sync(0xffffffffu, b, base + 8) << 16) |
                              (__shfl_sync(0xffffffffu, b, base + 12) << 24);
        const int chunk = 2 * seg + (base >> 4);
        if ((lane & 15u) == 0 && chunk * 128 < C)
          *reinterpret_cast<uint32_t*>(sc + (chunk * row_tiles + atom_row) * 512 + in_atom) = word;
      }
    }
  }
}

}  // namespace

size_t quantize_rows_smem_bytes(int E) { return sizeof(int) * (2 * static_cast<size_t>(E) + 3); }

cudaError_t launch_mxfp8_quantize_rows(const void* src, int src_rows, const int32_t* row_index,
                                       int M, int C, const int32_t* expert_off, int E, void* q,
                                       void* sc, long long Mcap, int rule, int* status,
                                       int num_sms, cudaStream_t stream) {
  const size_t smem = quantize_rows_smem_bytes(E);
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, mxfp8_quantize_rows_kernel, kRThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const long long rows_blocks = (Mcap + kRWarps - 1) / kRWarps;
  long long grid = static_cast<long long>(num_sms) * per_sm;
  if (grid > rows_blocks) grid = rows_blocks;
  if (grid < 1) grid = 1;
  mxfp8_quantize_rows_kernel<<<static_cast<unsigned>(grid), kRThreads, smem, stream>>>(
      static_cast<const uint16_t*>(src), src_rows, row_index, M, C, expert_off, E,
      static_cast<uint8_t*>(q), static_cast<uint8_t*>(sc), Mcap, rule, status);
  return cudaGetLastError();
}

}  // namespace mgw
