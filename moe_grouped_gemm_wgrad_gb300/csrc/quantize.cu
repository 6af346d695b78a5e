// MXFP8 quantization of a wgrad operand: bf16 [M, C] (token-major) -> e4m3
// [C, Mcap] (token-contiguous, per-expert 128-padded) + e8m0 scale atoms.
//
// HBM-bound transpose-quantize.  One work unit is 128 padded tokens x 128
// features.  A persistent grid walks the units; each CTA has two units' bf16
// tiles (32 KB each) in its input ring and refills a stage as soon as its values
// are in registers, so HBM reads overlap the conversion of the unit just read.  The
// lane that issues a stage's load also publishes the unit's token count with it, and
// the unit coordinates step with the grid stride, so a unit costs the consumers no
// search and no division.  Per unit every thread owns one pair of adjacent features
// and one 32-token block: 32-bit shared-memory reads, both block maxima at once with a
// packed bf16 magnitude max, an exact power-of-two scale applied by packed fp32x2
// multiplies, the hardware's round-to-nearest-even saturating e4m3 convert.  The e4m3
// tile (128B-swizzled) and its 512-byte scale atom leave through a double-buffered
// staging area with TMA bulk stores, so the CTA goes on to the next unit while they
// drain.
#include <cuda_bf16.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "mx.cuh"

namespace mgw {
namespace {

constexpr int kThreads = 256;
constexpr int kInBytes = 128 * 128 * 2;  // bf16 tile [token][feature], 256-byte rows
constexpr int kInStages = 2;
constexpr int kOutTile = 128 * 128;      // e4m3 tile [feature][token], 128B-swizzled rows
constexpr int kSf = 512;
constexpr int kOutBuf = 17408;           // tile + scale atom, padded to 1024 B
constexpr int kOffOut = kInStages * kInBytes;
constexpr int kOffBar = kOffOut + 2 * kOutBuf;
constexpr int kOffTable = kOffBar + 8 * kInStages + 16;
static_assert(kInStages <= 2, "misc area: flag, abort, one token count per stage");

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void bulk_store_1d(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(gdst)),
               "r"(ssrc), "r"(bytes)
               : "memory");
}
// Running largest magnitude of each bf16 half of m and v, lane by lane.  The sign of the
// result is meaningless (the caller clears it); a NaN in either input gives NaN, whose
// cleared bits, like any NaN's or an infinity's, carry the all-ones exponent.
__device__ __forceinline__ uint32_t amax_bf16x2(uint32_t m, uint32_t v) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(v));
  return r;
}
// Two fp32 products a*s, b*s in one packed multiply (each rounded as the scalar one).
__device__ __forceinline__ void mul_f32x2(uint32_t a, uint32_t b, uint64_t s2, float& x, float& y) {
  asm("{\n\t.reg .b64 t, r;\n\tmov.b64 t, {%2, %3};\n\tmul.rn.f32x2 r, t, %4;\n\t"
      "mov.b64 {%0, %1}, r;\n\t}"
      : "=f"(x), "=f"(y)
      : "r"(a), "r"(b), "l"(s2));
}
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

struct Unit {
  int valid;  // tokens of the chunk that belong to the expert (0: padding-only chunk)
  int row0;   // first source token
};

__device__ __forceinline__ Unit locate(int ch, int used_chunks, const int* s_off, const int* s_pad,
                                       int E) {
  Unit u{0, 0};
  if (ch < used_chunks) {
    // the largest e with P[e] <= 128*ch: always a non-empty expert for a used chunk
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
    u.valid = min(128, s_off[lo + 1] - s_off[lo] - tin);
    u.row0 = s_off[lo] + tin;
  }
  return u;
}

// kGather: token row t of the [M, C] source is row row_index[t] of the unpermuted token
// matrix [src_rows, C] (tm_src then has a one-row box); rows arrive four at a time with
// tile::gather4 TMA loads.  Otherwise the source is contiguous and each unit's rows
// arrive as one TMA tile.
template <bool kGather>
__global__ void __launch_bounds__(kThreads, 2) mxfp8_quantize_kernel(
    const __grid_constant__ CUtensorMap tm_src, const __grid_constant__ CUtensorMap tm_q, int M,
    int C, const int32_t* __restrict__ expert_off, int E, uint8_t* __restrict__ sc, long long Mcap,
    int rule, int* status, const uint16_t* __restrict__ gsrc, const int32_t* __restrict__ row_index,
    int src_rows) {
  extern __shared__ uint8_t smem_raw[];
  // 128B-swizzled TMA tiles want 1024-byte alignment; the launch adds the slack.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  // [0] flag [1] abort [2 + s] tokens of the expert in the unit loaded into stage s
  int* s_misc = reinterpret_cast<int*>(smem + kOffBar + 8 * kInStages);
  int* s_off = reinterpret_cast<int*>(smem + kOffTable);
  int* s_pad = s_off + (E + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&s_misc[1]);
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_misc[1] = 0;
    for (int s = 0; s < kInStages; ++s) mbar_init(sbase + kOffBar + 8 * s, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_src);
    tma_prefetch_desc(&tm_q);
  }
  if (!load_offsets(expert_off, E, M, s_off, s_pad, &s_misc[0], status)) return;

  const int col_tiles = C / 128;
  // below 2^31: q holds C x Mcap bytes, 16 KB per unit
  const int units = static_cast<int>((Mcap / 128) * col_tiles);
  const int used_chunks = s_pad[E] / 128;
  const int stride = gridDim.x;

  // Loads of unit u into input stage s, issued by warp 0 in two halves so that the
  // gather indices can be fetched early: prep() resolves the unit (and, for a gathered
  // source, loads its row indices into registers), fire() issues the copies.
  // Contiguous: one TMA tile (rows past the expert are read but masked; rows past M come
  // back as zeros).  Gather: lane l brings rows 4l .. 4l+3 with one tile::gather4 TMA;
  // indices outside [0, src_rows) and rows past the expert's last token are passed as
  // row -1, an out-of-bounds coordinate the TMA fills with zeros (bad indices also set
  // kDevBadIndex).  Padding-only units load nothing.
  const uint32_t lane = lane_id();
  struct Pending {
    int ct, valid, bad;
    int rr[4];
  };
  auto prep = [&](int u) {
    Pending pd;
    const int ch = u / col_tiles;
    pd.ct = u % col_tiles;
    const Unit un = locate(ch, used_chunks, s_off, s_pad, E);
    pd.valid = un.valid;
    pd.bad = 0;
    pd.rr[0] = un.row0;
    if (kGather) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = 4 * static_cast<int>(lane) + j;
        int idx = -1;
        if (r < un.valid) {
          idx = row_index[un.row0 + r];
          if (idx < 0 || idx >= src_rows) {
            idx = -1;
            pd.bad = 1;
          }
        }
        pd.rr[j] = idx;
      }
    }
    return pd;
  };
  auto fire = [&](const Pending& pd, int s) {
    const uint32_t bar = sbase + kOffBar + 8 * s;
    // published to the consumers by the arrive's release
    if (lane == 0) s_misc[2 + s] = pd.valid;
    if (!kGather) {
      if (lane != 0) return;
      if (pd.valid > 0) {
        mbar_arrive_expect_tx(bar, kInBytes);
        tma_load_2d(sbase + s * kInBytes, &tm_src, pd.ct * 128, pd.rr[0], bar);
      } else {
        mbar_arrive(bar);
      }
      return;
    }
    if (pd.valid <= 0) {
      if (lane == 0) mbar_arrive(bar);
      return;
    }
    const int groups = (pd.valid + 3) >> 2;
    const int bad = __any_sync(0xffffffffu, pd.bad);
    if (lane == 0) {
      if (bad && status) atomicOr(status, kDevBadIndex);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(groups) * 1024u);
    }
    __syncwarp();
    if (static_cast<int>(lane) < groups) {
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(sbase + s * kInBytes + lane * 1024u),
          "l"(reinterpret_cast<uint64_t>(&tm_src)), "r"(pd.ct * 128), "r"(pd.rr[0]), "r"(pd.rr[1]),
          "r"(pd.rr[2]), "r"(pd.rr[3]), "r"(bar)
          : "memory");
    }
  };
  if (tid < 32) {
    for (int s = 0; s < kInStages; ++s) {
      const int u = static_cast<int>(blockIdx.x) + s * stride;
      if (u < units) fire(prep(u), s);
    }
  }

  const int p = tid & 63;   // feature pair: features 2p, 2p+1 of the tile
  const int kb = tid >> 6;  // 32-token block of the chunk
  uint32_t phase = 0;
  int stage = 0, ob = 0;
  // (chunk, column tile) of unit u, stepped by the grid stride without a division per unit
  const int step_ch = stride / col_tiles, step_ct = stride % col_tiles;
  int ch = static_cast<int>(blockIdx.x) / col_tiles, ct = static_cast<int>(blockIdx.x) % col_tiles;
  for (int u = blockIdx.x; u < units; u += stride) {
    // Every thread waits; the decision to give up is made uniformly for the block.
    const int timed_out = mbar_wait(sbase + kOffBar + 8 * stage, phase, abort_flag) ? 0 : 1;
    if (__syncthreads_or(timed_out)) {
      // Only reachable if a TMA load never lands; report and stop this CTA's work.
      if (tid == 0) {
        if (status) atomicOr(status, kDevTimeout);
        *abort_flag = 1;
      }
      break;
    }
    const int valid = s_misc[2 + stage];
    // the unit that will refill this stage: resolve it (and load its indices) now
    const int nu = u + kInStages * stride;
    Pending next{0, 0, 0, {0, 0, 0, 0}};
    if (tid < 32 && nu < units) next = prep(nu);
    const uint32_t* in = reinterpret_cast<const uint32_t*>(smem + stage * kInBytes) + kb * 32 * 64 + p;
    uint32_t v[32];
    uint32_t amax = 0;  // block maxima: feature 2p in the low half, 2p+1 in the high half
    if (valid >= 128) {  // the same branch for the whole CTA
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = in[i * 64];  // bf16 pair (2p low, 2p+1 high)
        amax = amax_bf16x2(amax, v[i]);
      }
    } else {
      const int nvalid = min(32, max(0, valid - kb * 32));
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = (i < nvalid) ? in[i * 64] : 0u;
        amax = amax_bf16x2(amax, v[i]);
      }
    }
    amax &= 0x7FFF7FFFu;  // |bf16| orders like its bits
    // Every value of the stage went into the block maxima, so the stage is read: refill it
    // now, and the load overlaps this unit's conversion.
    __syncthreads();
    if (tid < 32 && nu < units) fire(next, stage);
    float inv_lo, inv_hi;
    int byte_lo = scale_byte(amax & 0xFFFFu, rule, &inv_lo);
    int byte_hi = scale_byte(amax >> 16, rule, &inv_hi);
    if (valid <= kb * 32) byte_lo = byte_hi = 0;  // a block with no token of the expert: padding
    const uint64_t s_lo = (static_cast<uint64_t>(__float_as_uint(inv_lo)) << 32) | __float_as_uint(inv_lo);
    const uint64_t s_hi = (static_cast<uint64_t>(__float_as_uint(inv_hi)) << 32) | __float_as_uint(inv_hi);
    uint32_t pl[8], ph[8];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      float a0, a1, a2, a3, b0, b1, b2, b3;
      mul_f32x2(v[i] << 16, v[i + 1] << 16, s_lo, a0, a1);
      mul_f32x2(v[i + 2] << 16, v[i + 3] << 16, s_lo, a2, a3);
      mul_f32x2(v[i] & 0xFFFF0000u, v[i + 1] & 0xFFFF0000u, s_hi, b0, b1);
      mul_f32x2(v[i + 2] & 0xFFFF0000u, v[i + 3] & 0xFFFF0000u, s_hi, b2, b3);
      pl[i / 4] = cvt_e4m3x4(a0, a1, a2, a3);
      ph[i / 4] = cvt_e4m3x4(b0, b1, b2, b3);
    }
    // The store issued from this output buffer two units ago must have read it.
    if (tid == 0) bulk_wait_read1();
    __syncthreads();  // output buffer `ob` free
    {
      // 128 feature rows x 128 token bytes, 16-byte chunk j of row r at (j ^ (r % 8)).
      const uint32_t obase = sbase + kOffOut + ob * kOutBuf;
      const int r0 = 2 * p, r1 = 2 * p + 1;
      const uint32_t a0 = obase + r0 * 128, a1 = obase + r1 * 128;
      st_shared_v4(a0 + (((2 * kb) ^ (r0 & 7)) << 4), pl[0], pl[1], pl[2], pl[3]);
      st_shared_v4(a0 + (((2 * kb + 1) ^ (r0 & 7)) << 4), pl[4], pl[5], pl[6], pl[7]);
      st_shared_v4(a1 + (((2 * kb) ^ (r1 & 7)) << 4), ph[0], ph[1], ph[2], ph[3]);
      st_shared_v4(a1 + (((2 * kb + 1) ^ (r1 & 7)) << 4), ph[4], ph[5], ph[6], ph[7]);
      uint8_t* s_sf = smem + kOffOut + ob * kOutBuf + kOutTile;
      s_sf[(r0 & 31) * 16 + (r0 >> 5) * 4 + kb] = static_cast<uint8_t>(byte_lo);
      s_sf[(r1 & 31) * 16 + (r1 >> 5) * 4 + kb] = static_cast<uint8_t>(byte_hi);
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      const uint32_t obase = sbase + kOffOut + ob * kOutBuf;
      tma_store_2d(&tm_q, ch * 128, ct * 128, obase);
      bulk_store_1d(sc + (static_cast<size_t>(ch) * col_tiles + ct) * kSf, obase + kOutTile, kSf);
      bulk_commit();
    }
    ob ^= 1;
    if (++stage == kInStages) stage = 0, phase ^= 1u;
    ct += step_ct;
    ch += step_ch;
    if (ct >= col_tiles) ct -= col_tiles, ++ch;
  }
  // All bulk stores complete before the CTA exits; loads issued for units this CTA never
  // reached (only after an abort) must land too.
  if (tid == 0) bulk_wait0();
  __syncthreads();
  if (tid == 0 && *abort_flag) {
    int never = 0;
    for (int s = 0; s < kInStages; ++s) (void)mbar_wait(sbase + kOffBar + 8 * s, phase, &never);
  }
}

}  // namespace

size_t quantize_smem_bytes(int E) {
  return static_cast<size_t>(kOffTable) + sizeof(int) * (2 * (E + 1)) + 1024;
}

cudaError_t launch_mxfp8_quantize(const CUtensorMap& tm_src, const CUtensorMap& tm_q, int M,
                                  int C, const int32_t* expert_off, int E, void* sc,
                                  long long Mcap, int rule, int* status, int num_sms,
                                  cudaStream_t stream, const void* gsrc,
                                  const int32_t* row_index, int src_rows) {
  const size_t smem = quantize_smem_bytes(E);
  static thread_local uint64_t attr_ctx[2] = {0, 0};
  cudaError_t err = set_smem_attr_once(reinterpret_cast<const void*>(mxfp8_quantize_kernel<false>),
                                       quantize_smem_bytes(kMaxExperts), &attr_ctx[0]);
  if (err != cudaSuccess) return err;
  err = set_smem_attr_once(reinterpret_cast<const void*>(mxfp8_quantize_kernel<true>),
                           quantize_smem_bytes(kMaxExperts), &attr_ctx[1]);
  if (err != cudaSuccess) return err;
  const bool gather = row_index != nullptr;
  auto kernel = gather ? mxfp8_quantize_kernel<true> : mxfp8_quantize_kernel<false>;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const long long units = (Mcap / 128) * (C / 128);
  if (units > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  long long grid = static_cast<long long>(num_sms) * per_sm;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(
      tm_src, tm_q, M, C, expert_off, E, static_cast<uint8_t*>(sc), Mcap, rule, status,
      static_cast<const uint16_t*>(gsrc), row_index, src_rows);
  return cudaGetLastError();
}

}  // namespace mgw
