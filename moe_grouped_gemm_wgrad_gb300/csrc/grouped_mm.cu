// Grouped MXFP8 GEMM over routed rows (M-grouped) on tcgen05 tensor cores:
//
//   out[r, j] = sum_l A[r, l] * B_e(r)[j, l]
//
// the forward y = x W[e]^T (l = hidden) and the data gradient dx = dy W[e] (l = the
// expert's output features), both with operands quantized along l.  A is row-wise
// quantized on the padded row axis (expert e's rows from P[e], a multiple of 128), so
// a 128-row tile never mixes experts.  B_e is the expert's block of one quantized
// matrix [RB, LB]: rows from e * b_row_step, contraction columns from e * b_col_step
// (the forward's W stacked [E*N, K]: row step N; the data gradient's W^T quantized
// along n per expert, [K, E*N + pad]: column step N).
//
// Work item = (128-row tile of the padded row axis, 256-column output tile); every
// item runs the full contraction, so the items cost the same and a persistent grid of
// one CTA per SM takes them in order with a fixed stride (neighbouring CTAs share the
// A tile and the expert's B block in L2).
//
// Roles (320 threads):
//   warp 0      TMA producer: per 128-element contraction chunk, the A tile 128x128 B,
//               the B tile 256x128 B (both 128B-swizzled) and the two scale-atom sets
//               (512 B + 1 KB) into a 4-stage shared-memory ring.
//   warp 1      MMA issuer: scale atoms to TMEM (tcgen05.cp 32x128b.warpx4) one chunk
//               ahead, four block-scaled tcgen05.mma.kind::mxf8f6f4 (M=128, N=256,
//               K=32) per chunk, commit of the stage back to the producer.
//   warps 2-9   epilogue: drain the 128x256 fp32 accumulator from TMEM, release it,
//               round to bf16 and write the tile as four 128x64 boxes through one 16 KB
//               128B-swizzled staging tile: a TMA store when all 128 rows belong to the
//               expert, else coalesced 16-byte stores of the expert's rows only (the
//               rows past its last one belong to the next expert's tile).
#include <cuda_bf16.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace mgw {
namespace {

constexpr int BM = 128;  // rows per tile (MMA M)
constexpr int BN = 256;  // output columns per tile (MMA N)
constexpr int BL = 128;  // contraction elements per pipeline stage (four 32-element blocks)
constexpr int kStages = 4;
constexpr int kABytes = BM * BL;                // 16 KB
constexpr int kBBytes = BN * BL;                // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 48 KB, 1024-aligned
constexpr int kSfStage = 512 + 1024;            // SFA atom + two SFB atoms
constexpr int kOutBytes = BM * 64 * 2;          // bf16 staging: one 128 x 64 box
constexpr int kOffOut = kStages * kStageBytes;
constexpr int kOffSf = kOffOut + kOutBytes;
constexpr int kOffBar = kOffSf + kStages * kSfStage;
constexpr int kNumBars = 2 * kStages + 3;  // full[], empty[], acc_full, acc_empty, done
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffTable = kOffMisc + 16;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;  // scale slots: 16 TMEM columns per stage

__host__ __device__ constexpr size_t mm_smem_bytes(int E) {
  return static_cast<size_t>(kOffTable) + sizeof(int) * (2 * static_cast<size_t>(E) + 2) + 1024;
}
static_assert(mm_smem_bytes(kMaxExperts) <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_f32, uint32_t hi_f32) {
  const __nv_bfloat162 v =
      __floats2bfloat162_rn(__uint_as_float(lo_f32), __uint_as_float(hi_f32));
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  int never = 0;
  (void)mbar_wait(bar, parity, &never);
}

// Row tile t (padded rows 128t ..) -> its expert and the tile's first routed row.
struct Tile {
  int e;       // expert
  int row0;    // first routed row (expert_off[e] + 128t - P[e])
  int nrows;   // rows of the tile that belong to the expert (1..128)
};

__device__ __forceinline__ Tile locate_tile(int t, const int* s_off, const int* s_pad, int E) {
  const int p0 = t * BM;
  int lo = 0, hi = E - 1;  // the largest e with P[e] <= p0: a non-empty expert for a used tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pad[mid] <= p0)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int i0 = p0 - s_pad[lo];
  Tile tl;
  tl.e = lo;
  tl.row0 = s_off[lo] + i0;
  tl.nrows = min(BM, s_off[lo + 1] - s_off[lo] - i0);
  return tl;
}

__global__ void __launch_bounds__(kThreads, 1) grouped_mm_mxfp8_kernel(const __grid_constant__ MmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int E = args.E;
  int* s_misc = reinterpret_cast<int*>(smem + kOffMisc);  // [0] tmem base [1] abort [2] flag
  int* s_off = reinterpret_cast<int*>(smem + kOffTable);
  int* s_pad = s_off + (E + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&s_misc[1]);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane = lane_id();

  if (tid == 0) s_misc[1] = 0;
  if (!load_offsets(args.expert_off, E, args.M, s_off, s_pad, &s_misc[2], args.status)) return;

  const uint32_t bar0 = sbase + kOffBar;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t bar_acc_full = bar0 + 8u * (2 * kStages);
  const uint32_t bar_acc_empty = bar0 + 8u * (2 * kStages + 1);
  const uint32_t bar_done = bar0 + 8u * (2 * kStages + 2);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, kEpiWarps);
    mbar_init(bar_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&args.tm_a);
    tma_prefetch_desc(&args.tm_b);
    tma_prefetch_desc(&args.tm_out);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_misc[0]), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(s_misc[0]);

  const int tiles_j = args.J / BN;
  const int nch = args.L / BL;
  const long long row_tiles = s_pad[E] / BM;
  const long long total = row_tiles * tiles_j;
  const long long a_tiles = args.Mcap / BM;  // row tiles of A's scale layout
  const long long b_tiles = args.RB / 128;   // row tiles of B's scale layout
  const long long first = blockIdx.x, step = gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int pending[kStages];
      uint32_t pending_phase[kStages];
      for (int s = 0; s < kStages; ++s) pending[s] = 0, pending_phase[s] = 0;
      bool ok = true;
      for (long long it = first; it < total && ok; it += step) {
        const int t = static_cast<int>(it / tiles_j);
        const int jt = static_cast<int>(it % tiles_j);
        const Tile tl = locate_tile(t, s_off, s_pad, E);
        const long long brow = static_cast<long long>(tl.e) * args.b_row_step + jt * BN;
        const long long bcol = static_cast<long long>(tl.e) * args.b_col_step;
        for (int c = 0; c < nch; ++c) {
          if (!mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full(stage);
          mbar_arrive_expect_tx(fb, kStageBytes + kSfStage);
          const uint32_t sa = sbase + stage * kStageBytes;
          tma_load_2d(sa, &args.tm_a, c * BL, t * BM, fb);
          tma_load_2d(sa + kABytes, &args.tm_b, static_cast<int>(bcol + c * BL),
                      static_cast<int>(brow), fb);
          const uint32_t ssf = sbase + kOffSf + stage * kSfStage;
          bulk_load(ssf, args.as + (c * a_tiles + t) * 512, 512, fb);
          bulk_load(ssf + 512, args.bs + ((bcol / 128 + c) * b_tiles + brow / 128) * 512, 1024, fb);
          pending[stage] = 1;
          pending_phase[stage] = phase;
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        if (args.status) atomicOr(args.status, kDevTimeout);
      }
      // Never leave the CTA with copies still landing in shared memory.
      for (int s = 0; s < kStages; ++s)
        if (pending[s]) mbar_wait_drain(bar_full(s), pending_phase[s]);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      // Waits for the chunk in `st` and copies its scale atoms to the stage's TMEM slot,
      // one chunk ahead of that chunk's MMAs.
      const uint64_t a_desc0 = sdesc_kmajor_sw128(sbase);
      const uint64_t sf_desc0 = make_sdesc(sbase + kOffSf, 0, 128, 0);
      auto stage_scales = [&](int st, uint32_t ph) -> bool {
        if (!mbar_wait(bar_full(st), ph, abort_flag)) return false;
        tc_fence_after();
        const uint64_t d = sf_desc0 + static_cast<uint32_t>(st * (kSfStage >> 4));
        const uint32_t tsf = tmem + kSfCol0 + 16u * st;
        tmem_cp_32x128b_warpx4(tsf, d);
        tmem_cp_32x128b_warpx4(tsf + 8, d + (512 >> 4));
        tmem_cp_32x128b_warpx4(tsf + 12, d + (1024 >> 4));
        return true;
      };
      for (long long it = first; it < total && ok; it += step) {
        if (!stage_scales(stage, phase) || !mbar_wait(bar_acc_empty, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int c = 0; c < nch; ++c) {
          const uint32_t tsf = tmem + kSfCol0 + 16u * stage;
          const uint64_t ad = a_desc0 + static_cast<uint32_t>(stage * (kStageBytes >> 4));
          mma_mxf8_chunk128<BM, BN>(tmem, ad, ad + (kABytes >> 4), tsf, tsf + 8, c != 0);
          // release the stage as soon as its MMAs are issued, then prepare the next one
          mma_commit(bar_empty(stage));
          if (++stage == kStages) stage = 0, phase ^= 1u;
          if (c + 1 < nch && !stage_scales(stage, phase)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        mma_commit(bar_acc_full);
        acc_phase ^= 1u;
      }
      if (!ok) {
        *abort_flag = 1;
        if (args.status) atomicOr(args.status, kDevTimeout);
      }
      mma_commit(bar_done);
      mbar_wait_drain(bar_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int half = ew >> 2;      // output columns [128*half, 128*half + 128)
    const int row = quarter * 32 + static_cast<int>(lane);
    const bool leader = (ew == 0 && lane == 0);
    const int etid = tid - 64;     // 0..255
    uint32_t acc_phase = 0;
    uint8_t* out = static_cast<uint8_t*>(args.out);
    const size_t pitch = static_cast<size_t>(args.J) * 2;
    for (long long it = first; it < total; it += step) {
      const int t = static_cast<int>(it / tiles_j);
      const int jt = static_cast<int>(it % tiles_j);
      const Tile tl = locate_tile(t, s_off, s_pad, E);
      uint32_t pk[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) pk[j] = 0u;
      if (!*abort_flag) {
        if (mbar_wait(bar_acc_full, acc_phase, abort_flag)) {
          tc_fence_after();
          uint32_t r[128];
          const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 128u * half;
          tmem_ld_32x32b_x32(ta + 0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          tmem_ld_32x32b_x32(ta + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          tmem_ld_32x32b_x32(ta + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
          tmem_ld_32x32b_x32(ta + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acc_empty);
#pragma unroll
          for (int j = 0; j < 64; ++j) pk[j] = pack_bf16x2(r[2 * j], r[2 * j + 1]);
        } else {
          *abort_flag = 1;
          if (lane == 0 && args.status) atomicOr(args.status, kDevTimeout);
        }
        acc_phase ^= 1u;
      }
      const bool full = tl.nrows == BM;
      const uint32_t stage_base = sbase + kOffOut;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (leader) bulk_wait_read0();  // the previous box has left the staging tile
        named_bar_sync(1, kEpiWarps * 32);
        if ((b >> 1) == half) {
#pragma unroll
          for (int chunk = 0; chunk < 8; ++chunk) {
            const int jj = (b & 1) * 8 + chunk;
            const uint32_t addr = stage_base + row * 128 + ((chunk ^ (row & 7)) << 4);
            st_shared_v4(addr, pk[4 * jj], pk[4 * jj + 1], pk[4 * jj + 2], pk[4 * jj + 3]);
          }
          fence_async_smem();
        }
        named_bar_sync(1, kEpiWarps * 32);
        if (*abort_flag) continue;
        if (full) {
          if (leader) {
            tma_store_2d(&args.tm_out, jt * BN + 64 * b, tl.row0, stage_base);
            bulk_commit();
          }
        } else {
          // 8 threads per 128-byte row segment, 32 rows per pass
          const int chunk = etid & 7;
#pragma unroll
          for (int pass = 0; pass < 4; ++pass) {
            const int rr = pass * 32 + (etid >> 3);
            if (rr < tl.nrows) {
              const uint4 v = ld_shared_v4(stage_base + rr * 128 + ((chunk ^ (rr & 7)) << 4));
              *reinterpret_cast<uint4*>(out + static_cast<size_t>(tl.row0 + rr) * pitch +
                                        static_cast<size_t>(jt * BN + 64 * b + 8 * chunk) * 2) = v;
            }
          }
        }
      }
    }
    if (leader) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_grouped_mm_mxfp8(const MmArgs& a, int num_sms, cudaStream_t stream) {
  static thread_local uint64_t attr_ctx = 0;
  cudaError_t err = set_smem_attr_once(reinterpret_cast<const void*>(grouped_mm_mxfp8_kernel),
                                       mm_smem_bytes(kMaxExperts), &attr_ctx);
  if (err != cudaSuccess) return err;
  // Upper bound on the used row tiles (the exact count is known on the device only).
  const long long max_tiles = a.Mcap / BM;
  const long long total = max_tiles * (a.J / BN);
  long long grid = num_sms;
  if (grid > total) grid = total;
  if (grid < 1) grid = 1;
  grouped_mm_mxfp8_kernel<<<static_cast<unsigned>(grid), kThreads, mm_smem_bytes(a.E), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mgw
