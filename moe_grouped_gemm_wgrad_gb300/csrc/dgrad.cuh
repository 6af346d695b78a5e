// Device helpers shared by the two grouped fp32 dgrad kernels (dgrad.cu: one SM per
// 128 x 256 output tile; dgrad_pair.cu: CTA pairs per 256 x 256 tile).
//
// Both compute dx[r, k] = sum_n dy[r, n] * W[e(r), n, k] with 3xTF32 tcgen05 MMAs: each fp32
// operand x is split as hi = tf32(x), lo = x - hi (tf32_split) and the product is
// hi*hi + hi*lo + lo*hi accumulated in fp32 in TMEM (Ootomo & Yokota, "Recovering single
// precision accuracy from Tensor Cores while surpassing the FP32 theoretical peak
// performance", IJHPCA 2022).  Both stage the operands the same way:
//   * raw chunks of 32 reduction elements n arrive by TMA: W[e] rows n (k contiguous,
//     unswizzled) and dy rows (n contiguous, 128B-swizzled, 128 rows per CTA);
//   * per 16-wide half of a chunk the transform warps read W column-wise and write the MMA's
//     B operand transposed (K-major, 128B-swizzled rows of 128 bytes: hi tf32 of the 16 n in
//     bytes 0-63, lo in 64-127), and read dy row-wise and store its hi/lo A operand columns
//     into TMEM (16 hi columns, then 16 lo columns);
//   * per half, 2 K-steps x 3 tcgen05.mma.kind::tf32 with A from TMEM.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "diag.cuh"
#include "kernels.h"

namespace mgw {
namespace dgrad {

constexpr int BK = 32;    // reduction (out_features) per raw chunk: one 128-byte row of fp32
constexpr int BKH = 16;   // reduction per operand stage (half a chunk)
constexpr int kRowsPerCta = 128;            // A rows (dx rows) per CTA: the TMEM lanes
constexpr int kRawDy = kRowsPerCta * BK * 4;  // raw dy rows per CTA and chunk: 16 KB

// 3xTF32 operand split: hi is x rounded to tf32 (10 stored mantissa bits), to nearest with ties
// away from zero, done on the sign-magnitude bits: add half the weight of the 13 dropped bits,
// then clear them.  lo = x - hi is exact in fp32 (|x - hi| <= 2^-11 |x|, and hi lies within a
// factor 2 of x), and it is handed to the tensor core as it is: reading it as tf32 drops or
// rounds its low 13 bits, an error of at most 2^-10 |lo| <= 2^-21 |x|.  Integer and fp32 adds
// only, no conversion instruction: the conversions' lower throughput bounded the transform
// warps.
__device__ __forceinline__ void tf32_split(float x, uint32_t& hi, uint32_t& lo) {
  hi = (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}

// Brings a tile of a tensor map into L2 only (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* m, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1)
               : "memory");
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, const uint32_t (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_global_v8(float* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  int never = 0;
  (void)mbar_wait(bar, parity, &never);
}

// The A half of one operand stage, for the thread of TMEM lane quarter q and 4-column group
// kh: dy[r][16h + 4kh .. +3] of row r = 32q + lane, read from the raw 128B-swizzled dy tile
// (a warp reads 32 rows at one logical 16-byte chunk, which the swizzle spreads over all
// banks) ...
__device__ __forceinline__ float4 load_a(uint32_t raw_dy, int h, uint32_t q, uint32_t lane, int kh) {
  const uint32_t r = q * 32u + lane;
  return ld_shared_f4(raw_dy + r * 128u + (((4u * h + kh) ^ (r & 7u)) << 4));
}
// ... split and stored as TMEM columns acol + 4kh (hi) and acol + 16 + 4kh (lo).
__device__ __forceinline__ void store_a(float4 a, uint32_t q, int kh, uint32_t tmem, uint32_t acol) {
  uint32_t ah[4], al[4];
  tf32_split(a.x, ah[0], al[0]);
  tf32_split(a.y, ah[1], al[1]);
  tf32_split(a.z, ah[2], al[2]);
  tf32_split(a.w, ah[3], al[3]);
  const uint32_t ta = tmem + (q * 32u << 16) + acol + 4u * kh;
  tmem_st_x4(ta, ah);
  tmem_st_x4(ta + 16, al);
}

// Stores the ncols accumulator columns of the rows of TMEM lane quarter `quarter` that hold dx
// rows row0 .. row0 + valid - 1 (valid may be <= 0) at dx columns col0 .., 32 columns per
// TMEM load.  Warp-uniform: all lanes of the warp call it with the same arguments.
__device__ __forceinline__ void store_acc_rows(const DgradArgs& args, uint32_t tmem, int quarter,
                                               uint32_t lane, int row0, int valid, int col0,
                                               int ncols) {
  if (quarter * 32 >= valid) return;
  if (!MGW_DIAG_CHECK(row0 >= 0 && row0 + valid <= args.rows && col0 >= 0 && col0 + ncols <= args.in_f,
                      lane == 0 ? args.status : nullptr))
    return;
  const int r = quarter * 32 + static_cast<int>(lane);
  float* dst = args.dx + static_cast<size_t>(row0 + (r < valid ? r : 0)) * args.in_f + col0;
  const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
  for (int j = 0; j < ncols / 32; ++j) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(ta + 32u * j, v);
    tmem_wait_ld();
    if (r < valid) {
      if (args.dx_align32) {
        // whole 32-byte sectors per store
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) st_global_v8(dst + 32 * j + 8 * qq, v + 8 * qq);
      } else {
#pragma unroll
        for (int qq = 0; qq < 8; ++qq)
          *reinterpret_cast<float4*>(dst + 32 * j + 4 * qq) =
              make_float4(__uint_as_float(v[4 * qq]), __uint_as_float(v[4 * qq + 1]),
                          __uint_as_float(v[4 * qq + 2]), __uint_as_float(v[4 * qq + 3]));
      }
    }
  }
}

// Item it -> (expert, row tile in the expert, k tile) via the prefix s_tp of per-expert row-tile
// counts (E + 1 entries); consecutive items share the row tile and step the k tile.
struct Item {
  int e, rt, kt;
};
__device__ __forceinline__ Item decode_item(long long it, int tiles_k, const int* s_tp, int E) {
  const int t = static_cast<int>(it / tiles_k);
  Item r;
  r.kt = static_cast<int>(it % tiles_k);
  int lo = 0, hi = E - 1;  // largest e with s_tp[e] <= t (a non-empty expert)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tp[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  r.e = lo;
  r.rt = t - s_tp[lo];
  return r;
}

}  // namespace dgrad
}  // namespace mgw
