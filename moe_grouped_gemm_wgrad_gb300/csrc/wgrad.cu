// Grouped MXFP8 expert weight gradient on tcgen05 tensor cores.
//
//   grad_w[e*N + n, k] = sum_{t in expert e} g[t, n] * x[t, k]
//
// Work item = (expert, 128-row N tile, 256-column K tile); one item's output tile
// is a 128 x 256 fp32 accumulator in TMEM (256 columns).  A persistent grid of one
// CTA per SM walks the items in a snake order over the experts sorted by descending
// token count (LPT), so the largest experts are spread first; experts with no tokens
// become store-only items that write zero rows.
//
// Roles (352 threads):
//   warp 0      TMA producer: per 128-token chunk, g^T tile 128x128 B, x^T tile
//               256x128 B (both 128B-swizzled) and the two e8m0 scale-factor atom
//               sets (512 B + 1 KB) into a 4-stage shared-memory ring.
//   warp 1      MMA issuer: copies the chunk's scale atoms to TMEM (tcgen05.cp,
//               32x128b.warpx4) and issues one block-scaled
//               tcgen05.mma.kind::mxf8f6f4 (M=128, N=256, K=32) per 32-token block
//               that holds tokens, then commits the stage back to the producer.
//   warp 10     zero writer: stores the rows of experts without tokens with plain
//               vector stores, overlapping the MMA work (single-SM kernel).
//   warps 2-9   epilogue: drain the accumulator (each warp: its TMEM lane quarter,
//               one 128-column half) into registers, release TMEM at once so the
//               next item's MMAs start, then round to bf16 and TMA-store the tile as
//               four 128 x 64 boxes through one 16 KB 128B-swizzled staging tile
//               (one box at a time, so the ring can hold four 48 KB stages).
#include <cuda_bf16.h>

#include <cstdint>
#include <cstdlib>

#include "common.cuh"
#include "diag.cuh"
#include "kernels.h"

namespace mgw {

MGW_DIAG_TIMELINE_DEFINE(wgrad, 1)

namespace {

constexpr int BM = 128;  // grad_w rows per tile (MMA M)
constexpr int BN = 256;  // grad_w cols per tile (MMA N)
constexpr int BT = 128;  // tokens per pipeline stage (four 32-token scale blocks)
constexpr int kStages = 4;
constexpr int kABytes = BM * BT;                 // 16 KB
constexpr int kBBytes = BN * BT;                 // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;   // 48 KB, 1024-aligned
constexpr int kSfStage = 512 + 1024;             // SFA atom + two SFB atoms
constexpr int kOutBytes = BM * 64 * 2;           // bf16 staging: one 128 x 64 box (16 KB)
constexpr int kOffOut = kStages * kStageBytes;
constexpr int kOffSf = kOffOut + kOutBytes;
constexpr int kOffBar = kOffSf + kStages * kSfStage;
constexpr int kNumBars = 2 * kStages + 3;        // full[], empty[], acc_full, acc_empty, done
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffTable = kOffMisc + 16;
constexpr int kThreads = 352;
constexpr int kEpiWarps = 8;
constexpr int kZeroWarp = 10;  // single-SM kernel: writes the tiles of experts without tokens
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;  // scale slots: 16 TMEM columns per stage

// Tables: expert_off and padded starts (int, E+1 each), LPT order (uint16, E).
__host__ __device__ constexpr size_t wgrad_smem_bytes(int E) {
  return static_cast<size_t>(kOffTable) + sizeof(int) * (2 * static_cast<size_t>(E) + 2) +
         sizeof(uint16_t) * static_cast<size_t>(E) + 1024;
}
static_assert(wgrad_smem_bytes(kMaxExperts) <= 232448, "shared memory budget");

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

// Snake order over the LPT-sorted items: round r hands items to CTAs left to right when r is
// even and right to left when r is odd, so the heaviest items do not all land on the same
// CTAs.  Every role of a CTA walks the same sequence.
struct ItemIter {
  long long total, grid, round;
  int cta;
  __device__ __forceinline__ bool next(long long& it) {
    while (true) {
      const long long base = round * grid;
      if (base >= total) return false;
      const long long idx = base + ((round & 1) ? (grid - 1 - cta) : cta);
      ++round;
      if (idx < total) {
        it = idx;
        return true;
      }
    }
  }
};

// Waits without honouring the abort flag (used to drain in-flight async work).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  int never = 0;
  (void)mbar_wait(bar, parity, &never);
}

__global__ void __launch_bounds__(kThreads, 1) grouped_wgrad_kernel(const __grid_constant__ WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int E = args.E, N = args.N, K = args.K;
  int* s_misc = reinterpret_cast<int*>(smem + kOffMisc);  // [0] tmem base [1] abort [2] flag
  int* s_off = reinterpret_cast<int*>(smem + kOffTable);
  int* s_pad = s_off + (E + 1);
  uint16_t* s_order = reinterpret_cast<uint16_t*>(s_pad + (E + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&s_misc[1]);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane = lane_id();

  if (tid == 0) s_misc[1] = 0;
  if (!load_offsets(args.expert_off, E, args.M, s_off, s_pad, &s_misc[2], args.status)) return;

  // LPT order: experts by descending token count, ties by index.
  for (int e = tid; e < E; e += kThreads) {
    const int ce = s_off[e + 1] - s_off[e];
    int rank = 0;
    for (int j = 0; j < E; ++j) {
      const int cj = s_off[j + 1] - s_off[j];
      rank += (cj > ce) || (cj == ce && j < e);
    }
    s_order[rank] = static_cast<uint16_t>(e);
  }
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

  const int tiles_n = N / BM, tiles_k = K / BN;
  // Item indices fit in 32 bits (the C ABI checks E x tiles < 2^31), so the per-item decode
  // uses 32-bit divisions: the MMA thread runs it once per item.
  const int per_expert = tiles_n * tiles_k;
  const long long total = static_cast<long long>(per_expert) * E;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int pending[kStages];
      uint32_t pending_phase[kStages];
      for (int s = 0; s < kStages; ++s) pending[s] = 0, pending_phase[s] = 0;
      bool ok = true, dropped = false;
      ItemIter items{total, gridDim.x, 0, static_cast<int>(blockIdx.x)};
      long long it = 0;
      while (ok && items.next(it)) {
        const int e = s_order[static_cast<int>(it) / per_expert];
        const int tile = static_cast<int>(it) % per_expert;
        const int nt = tile / tiles_k, kt = tile % tiles_k;
        const int cnt = s_off[e + 1] - s_off[e];
        if (cnt == 0) continue;
        const int nch = (cnt + BT - 1) / BT;
        const int ch0 = s_pad[e] / BT;
        for (int c = 0; c < nch; ++c) {
          if (!mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full(stage);
          mbar_arrive_expect_tx(fb, kStageBytes + kSfStage);
          if (args.drop_first_load && !dropped) {  // test hook: this stage never fills
            dropped = true;
            pending[stage] = 1;
            pending_phase[stage] = phase;
            if (++stage == kStages) stage = 0, phase ^= 1u;
            continue;
          }
          const uint32_t sa = sbase + stage * kStageBytes;
          const int tok = (ch0 + c) * BT;
          tma_load_2d(sa, &args.tm_a, tok, nt * BM, fb);
          tma_load_2d(sa + kABytes, &args.tm_b, tok, kt * BN, fb);
          const uint32_t ssf = sbase + kOffSf + stage * kSfStage;
          bulk_load(ssf, args.gs + (static_cast<size_t>(ch0 + c) * tiles_n + nt) * 512, 512, fb);
          bulk_load(ssf + 512,
                    args.xs + (static_cast<size_t>(ch0 + c) * (K / 128) + 2 * kt) * 512, 1024, fb);
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
      // Waits for the chunk in `stage` to land and copies its scale atoms to the stage's
      // TMEM slot (32 rows x 16 B each, 8-row core matrices 128 B apart).  Issued one
      // chunk ahead of that chunk's MMAs so the copy overlaps the previous chunk's MMAs.
      // Descriptors of stage 0; stage s adds its byte offset / 16 to the start-address field
      // (the whole ring lies below 256 KB, so the 14-bit field never carries).
      const uint64_t a_desc0 = sdesc_kmajor_sw128(sbase);
      const uint64_t sf_desc0 = make_sdesc(sbase + kOffSf, 0, 128, 0);
      auto stage_scales = [&](int st, uint32_t ph) -> bool {
        if (!mbar_wait_spin(bar_full(st), ph, abort_flag)) return false;
        tc_fence_after();
        const uint64_t d = sf_desc0 + static_cast<uint32_t>(st * (kSfStage >> 4));
        const uint32_t tsf = tmem + kSfCol0 + 16u * st;
        tmem_cp_32x128b_warpx4(tsf, d);
        tmem_cp_32x128b_warpx4(tsf + 8, d + (512 >> 4));
        tmem_cp_32x128b_warpx4(tsf + 12, d + (1024 >> 4));
        return true;
      };
      ItemIter items{total, gridDim.x, 0, static_cast<int>(blockIdx.x)};
      long long it = 0;
      while (ok && items.next(it)) {
        const int e = s_order[static_cast<int>(it) / per_expert];
        const int cnt = s_off[e + 1] - s_off[e];
        if (cnt == 0) continue;
        const int nch = (cnt + BT - 1) / BT;
        const int full_chunks = cnt / BT;  // chunks whose four 32-token blocks all hold tokens
        // first chunk's scales go in while the epilogue still drains the accumulator
        if (!stage_scales(stage, phase) || !mbar_wait_spin(bar_acc_empty, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int c = 0; c < nch; ++c) {
          const uint32_t tsf = tmem + kSfCol0 + 16u * stage;
          const uint64_t ad = a_desc0 + static_cast<uint32_t>(stage * (kStageBytes >> 4));
          const uint64_t bd = ad + (kABytes >> 4);
          if (c < full_chunks) {
            mma_mxf8_chunk128<BM, BN>(tmem, ad, bd, tsf, tsf + 8, c != 0);
          } else {
            const int nkb = (cnt - c * BT + 31) / 32;
            for (int kb = 0; kb < nkb; ++kb) {
              mma_mxf8_block32(tmem, ad + 2 * kb, bd + 2 * kb, idesc_mxf8_e4m3(BM, BN, kb, kb),
                               tsf, tsf + 8, (c | kb) != 0);
            }
          }
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
      // All MMAs issued by this thread complete before TMEM is released.
      mma_commit(bar_done);
      mbar_wait_drain(bar_done, 0);
    }
  } else if (warp == kZeroWarp) {
    // ----------------------------------------- zero tiles of experts without tokens
    // Plain 16-byte stores (one 512-byte row segment per instruction) that overlap the
    // MMA work of the other roles instead of queueing behind it in the epilogue.
    uint8_t* out = static_cast<uint8_t*>(args.out);
    const size_t pitch = static_cast<size_t>(K) * 2;
    ItemIter items{total, gridDim.x, 0, static_cast<int>(blockIdx.x)};
    long long it = 0;
    while (items.next(it)) {
      const int e = s_order[static_cast<int>(it) / per_expert];
      if (s_off[e + 1] != s_off[e]) continue;
      const int tile = static_cast<int>(it) % per_expert;
      const int nt = tile / tiles_k, kt = tile % tiles_k;
      uint8_t* base = out + (static_cast<size_t>(e) * N + nt * BM) * pitch +
                      static_cast<size_t>(kt) * BN * 2 + lane * 16;
#pragma unroll 4
      for (int r = 0; r < BM; ++r)
        *reinterpret_cast<uint4*>(base + r * pitch) = make_uint4(0u, 0u, 0u, 0u);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int half = ew >> 2;      // output columns [128*half, 128*half + 128)
    const int row = quarter * 32 + static_cast<int>(lane);
    const bool leader = (ew == 0 && lane == 0);
    uint32_t acc_phase = 0;
    ItemIter items{total, gridDim.x, 0, static_cast<int>(blockIdx.x)};
    long long it = 0;
    while (items.next(it)) {
      const int e = s_order[static_cast<int>(it) / per_expert];
      const int tile = static_cast<int>(it) % per_expert;
      const int nt = tile / tiles_k, kt = tile % tiles_k;
      const int cnt = s_off[e + 1] - s_off[e];
      if (cnt == 0) continue;  // written by the zero warp
      uint32_t pk[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) pk[j] = 0u;
      if (cnt > 0 && !*abort_flag) {
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
      // Four 128 x 64 boxes go out through one 16 KB staging tile, one after another:
      // the warps of the box's column half write it (128B swizzle), one thread stores it.
      const uint32_t stage_base = sbase + kOffOut;
      const int orow = e * N + nt * BM;
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
        if (leader && !*abort_flag) {
          tma_store_2d(&args.tm_out, kt * BN + 64 * b, orow, stage_base);
          bulk_commit();
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



// ---------------------------------------------------------------------------
// CTA-pair kernel (two SMs per output tile, tcgen05 cta_group::2), used when N % 256 == 0.
//
// A pair of CTAs in a (2,1,1) cluster owns a 256 x 256 grad_w tile: CTA r holds rows
// 128r .. 128r+127 of the tile (its A operand, its TMEM accumulator) and columns
// 128r .. 128r+127 of the B operand; the even CTA issues one
// tcgen05.mma.cta_group::2.kind::mxf8f6f4 (M=256, N=256, K=32) per 32-token block, which
// reads A from each CTA's shared memory and B from both halves.  Per 128-token chunk each
// SM takes in 32 KB of operands by TMA instead of the single-SM tile's 48 KB for the same
// work per SM, which leaves room for a six-stage ring.
//
// Scale factors reach TMEM through four writer warps per CTA (one per TMEM lane quarter)
// with tcgen05.st, not through tcgen05.cp from the MMA-issuing thread: measured on GB300,
// the three copies per chunk cost that thread ~130 cycles per chunk in which the MMA pipe
// idles, and a burst of them per window costs the same per copy.  Each CTA's scale atoms
// land in its own stage slot (bulk copies counted on a local barrier); its writers place
// them in the stage's TMEM slot and report to the even CTA's sf_ready barrier.
//
// Roles (480 threads per CTA):
//   warp 0       TMA producer (both CTAs): its g^T rows and half of x^T per chunk, counted
//                on the even CTA's full barrier; its scale atoms on its own sf_full.
//   warp 1       MMA issuer (even CTA): per chunk waits full and sf_ready, issues four
//                pair MMAs, commits the stage back to both producers.
//   warps 2-9    epilogue (both CTAs): drain this CTA's accumulator, release it to the even
//                CTA, round to bf16, TMA-store 128 x 256 through one staging box.
//   warp 10      zero writer: this CTA's rows of the tiles of experts without tokens.
//   warps 11-14  scale writers (both CTAs): one TMEM lane quarter each.
//
// Barriers: the even CTA's commits are multicast to both CTAs' empty / accumulator-full
// barriers; both CTAs' epilogues and scale writers arrive on the even CTA's
// accumulator-empty and sf_ready barriers.  Each CTA's producer ends by waiting until every
// stage it filled has been released, so no copy is still landing when a CTA exits.
constexpr int kPStages = 6;
constexpr int kPABytes = 128 * BT;                  // 16 KB: this CTA's 128 rows of g^T
constexpr int kPBBytes = 128 * BT;                  // 16 KB: this CTA's half of x^T
constexpr int kPStageBytes = kPABytes + kPBBytes;   // 32 KB
constexpr int kPOffOut = kPStages * kPStageBytes;
constexpr int kPOffSf = kPOffOut + kOutBytes;
constexpr int kPOffBar = kPOffSf + kPStages * kSfStage;
// full[], empty[], sf_full[], sf_ready[], acc_full, acc_empty, done
constexpr int kPNumBars = 4 * kPStages + 3;
constexpr int kPOffMisc = (kPOffBar + kPNumBars * 8 + 15) & ~15;
constexpr int kPOffTable = kPOffMisc + 16;
constexpr int kSfWarp0 = 11;                        // scale writers: warps 11-14
constexpr int kPThreads = (kSfWarp0 + 4) * 32;      // 480

__host__ __device__ constexpr size_t wgrad_pair_smem_bytes(int E) {
  return static_cast<size_t>(kPOffTable) + sizeof(int) * (2 * static_cast<size_t>(E) + 2) +
         sizeof(uint16_t) * static_cast<size_t>(E) + 1024;
}
static_assert(wgrad_pair_smem_bytes(kMaxPairExperts) <= 232448, "shared memory budget");
static_assert(kSfCol0 + 16 * kPStages <= kTmemCols, "TMEM budget");

// The four pair MMAs (M=256, N=256, K=32 each) of one 128-token chunk, constant
// instruction descriptors, the K step as +2 in the descriptors' start-address field.
__device__ __forceinline__ void mma_mxf8_chunk128_pair(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                                       uint32_t sfa, uint32_t sfb,
                                                       uint32_t accumulate) {
  mma_mxf8_block32_pair(d, adesc, bdesc, idesc_mxf8_e4m3(256, 256, 0, 0), sfa, sfb, accumulate);
  mma_mxf8_block32_pair(d, adesc + 2, bdesc + 2, idesc_mxf8_e4m3(256, 256, 1, 1), sfa, sfb, 1u);
  mma_mxf8_block32_pair(d, adesc + 4, bdesc + 4, idesc_mxf8_e4m3(256, 256, 2, 2), sfa, sfb, 1u);
  mma_mxf8_block32_pair(d, adesc + 6, bdesc + 6, idesc_mxf8_e4m3(256, 256, 3, 3), sfa, sfb, 1u);
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c,
                                             uint32_t& d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr)
               : "memory");
}
// 32 lanes x 4 / 8 consecutive 32-bit columns from registers: thread i -> lane (base+i).
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, uint32_t a, uint32_t b,
                                                  uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    grouped_wgrad_pair_kernel(const __grid_constant__ WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int E = args.E, N = args.N, K = args.K;
  int* s_misc = reinterpret_cast<int*>(smem + kPOffMisc);  // [0] tmem base [1] abort [2] flag
  int* s_off = reinterpret_cast<int*>(smem + kPOffTable);
  int* s_pad = s_off + (E + 1);
  uint16_t* s_order = reinterpret_cast<uint16_t*>(s_pad + (E + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&s_misc[1]);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair MMAs
  const bool leader = rank == 0;

  if (tid == 0) s_misc[1] = 0;
  // Both CTAs read the same offsets, so both return here or neither does.
  if (!load_offsets(args.expert_off, E, args.M, s_off, s_pad, &s_misc[2], args.status)) return;

  for (int e = tid; e < E; e += kPThreads) {
    const int ce = s_off[e + 1] - s_off[e];
    int rank_e = 0;
    for (int j = 0; j < E; ++j) {
      const int cj = s_off[j + 1] - s_off[j];
      rank_e += (cj > ce) || (cj == ce && j < e);
    }
    s_order[rank_e] = static_cast<uint16_t>(e);
  }
  const uint32_t bar0 = sbase + kPOffBar;
  auto bar_full = [&](int st) { return bar0 + 8u * st; };                   // even CTA
  auto bar_empty = [&](int st) { return bar0 + 8u * (kPStages + st); };
  auto bar_sf_full = [&](int st) { return bar0 + 8u * (2 * kPStages + st); };
  auto bar_sf_ready = [&](int st) { return bar0 + 8u * (3 * kPStages + st); };  // even CTA
  const uint32_t bar_acc_full = bar0 + 8u * (4 * kPStages);
  const uint32_t bar_acc_empty = bar0 + 8u * (4 * kPStages + 1);           // even CTA
  const uint32_t bar_done = bar0 + 8u * (4 * kPStages + 2);
  if (tid == 0) {
    for (int st = 0; st < kPStages; ++st) {
      mbar_init(bar_full(st), 1);
      mbar_init(bar_empty(st), 1);
      mbar_init(bar_sf_full(st), 1);
      mbar_init(bar_sf_ready(st), 8);  // four writer warps in each CTA
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, 2 * kEpiWarps);
    mbar_init(bar_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&args.tm_a);
    tma_prefetch_desc(&args.tm_b);
    tma_prefetch_desc(&args.tm_out);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&s_misc[0]), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(s_misc[0]);
  // The peer CTA's abort flag: a role that gives up tells both CTAs.
  const uint32_t peer_abort = map_to_cta(smem_u32(&s_misc[1]), rank ^ 1u);
  auto abort_both = [&]() {
    *abort_flag = 1;
    st_cluster_u32(peer_abort, 1u);
    if (args.status) atomicOr(args.status, kDevTimeout);
  };

  const int pairs_n = N / 256, tiles_k = K / BN;
  const int per_expert = pairs_n * tiles_k;  // 32-bit: the C ABI checks E x tiles < 2^31
  const long long total = static_cast<long long>(per_expert) * E;
  const long long npairs = gridDim.x >> 1;
  const int pair = static_cast<int>(blockIdx.x >> 1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int filled[kPStages];
      uint32_t filled_phase[kPStages];
      for (int st = 0; st < kPStages; ++st) filled[st] = 0, filled_phase[st] = 0;
      bool ok = true;
      const uint32_t full0_leader = map_to_cta(bar_full(0), 0);
      ItemIter items{total, npairs, 0, pair};
      long long it = 0;
      while (ok && items.next(it)) {
        const int e = s_order[static_cast<int>(it) / per_expert];
        const int tile = static_cast<int>(it) % per_expert;
        const int np = tile / tiles_k, kt = tile % tiles_k;
        const int cnt = s_off[e + 1] - s_off[e];
        if (cnt == 0) continue;
        const int nch = (cnt + BT - 1) / BT;
        const int ch0 = s_pad[e] / BT;
        const int arow = np * 256 + 128 * static_cast<int>(rank);   // this CTA's g^T rows
        const int brow = kt * BN + 128 * static_cast<int>(rank);    // this CTA's x^T rows
        for (int c = 0; c < nch; ++c) {
          if (!mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(bar_full(stage), 2 * kPStageBytes);
          const uint32_t fb = full0_leader + 8u * stage;  // the even CTA's full barrier
          const uint32_t sa = sbase + stage * kPStageBytes;
          const int ch = ch0 + c;
          (void)MGW_DIAG_CHECK(static_cast<long long>(ch + 1) * BT <= args.mcap && arow + 128 <= N &&
                                   brow + 128 <= K,
                               args.status);
          tma_load_2d_pair(sa, &args.tm_a, ch * BT, arow, fb);
          tma_load_2d_pair(sa + kPABytes, &args.tm_b, ch * BT, brow, fb);
          // this CTA's g atom and both x atoms of the K tile (every CTA's accumulator spans
          // all 256 columns), counted on this CTA's own sf_full barrier
          const uint32_t sfb = bar_sf_full(stage);
          mbar_arrive_expect_tx(sfb, kSfStage);
          const uint32_t ssf = sbase + kPOffSf + stage * kSfStage;
          bulk_load(ssf, args.gs + (static_cast<size_t>(ch) * (N / 128) + arow / 128) * 512, 512, sfb);
          bulk_load(ssf + 512, args.xs + (static_cast<size_t>(ch) * (K / 128) + 2 * kt) * 512, 1024, sfb);
          filled[stage] = 1;
          filled_phase[stage] = phase;
          if (++stage == kPStages) stage = 0, phase ^= 1u;
        }
      }
      if (!ok) abort_both();
      // Every stage this CTA filled is released by the MMAs that read it (or, after an
      // abort, the wait gives up after its time limit, long after any copy has landed).
      for (int st = 0; st < kPStages; ++st)
        if (filled[st]) mbar_wait_drain(bar_empty(st), filled_phase[st]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer (even CTA only)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      constexpr uint16_t kBoth = 0x3;
      const uint64_t a_desc0 = sdesc_kmajor_sw128(sbase);
      ItemIter items{total, npairs, 0, pair};
      long long it = 0;
      while (ok && items.next(it)) {
        const int e = s_order[static_cast<int>(it) / per_expert];
        const int cnt = s_off[e + 1] - s_off[e];
        if (cnt == 0) continue;
        const int nch = (cnt + BT - 1) / BT;
        const int full_chunks = cnt / BT;
        if (!mbar_wait_spin(bar_acc_empty, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        for (int c = 0; c < nch; ++c) {
          // operands in both CTAs, scale factors in both CTAs' TMEM
          if (!mbar_wait_spin(bar_full(stage), phase, abort_flag) ||
              !mbar_wait_spin(bar_sf_ready(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tsf = tmem + kSfCol0 + 16u * stage;
          const uint64_t ad = a_desc0 + static_cast<uint32_t>(stage * (kPStageBytes >> 4));
          const uint64_t bd = ad + (kPABytes >> 4);
          if (c < full_chunks) {
            mma_mxf8_chunk128_pair(tmem, ad, bd, tsf, tsf + 8, c != 0);
          } else {
            const int nkb = (cnt - c * BT + 31) / 32;
            for (int kb = 0; kb < nkb; ++kb)
              mma_mxf8_block32_pair(tmem, ad + 2 * kb, bd + 2 * kb, idesc_mxf8_e4m3(256, 256, kb, kb),
                                    tsf, tsf + 8, (c | kb) != 0);
          }
          mma_commit_pair(bar_empty(stage), kBoth);
          if (++stage == kPStages) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit_pair(bar_acc_full, kBoth);
        acc_phase ^= 1u;
      }
      if (!ok) abort_both();
      // All MMAs issued by this thread complete before TMEM is released.
      mma_commit_pair(bar_done, 0x1);
      mbar_wait_drain(bar_done, 0);
    }
  } else if (warp >= kSfWarp0) {
    // ----------------------------------- scale writers: TMEM lane quarter warp % 4
    // Atom row r0 (16 bytes: words r1 = 0..3, feature r0 + 32 r1, one byte per 32-token
    // block) goes to TMEM lane r0 of every lane quarter, column r1 of the stage's slot: the
    // layout tcgen05.mma reads scale factors from (the same bytes a 32x128b.warpx4 copy of
    // the atom places).
    const uint32_t quarter = static_cast<uint32_t>(warp & 3);
    const uint32_t sf_ready0 = map_to_cta(bar_sf_ready(0), 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    ItemIter items{total, npairs, 0, pair};
    long long it = 0;
    while (ok && items.next(it)) {
      const int e = s_order[static_cast<int>(it) / per_expert];
      const int cnt = s_off[e + 1] - s_off[e];
      if (cnt == 0) continue;
      const int nch = (cnt + BT - 1) / BT;
      for (int c = 0; c < nch; ++c) {
        if (!mbar_wait(bar_sf_full(stage), phase, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t ssf = sbase + kPOffSf + stage * kSfStage + 16u * lane;
        uint32_t a0, a1, a2, a3;
        uint32_t b[8];
        ld_shared_v4(ssf, a0, a1, a2, a3);
        ld_shared_v4(ssf + 512, b[0], b[1], b[2], b[3]);
        ld_shared_v4(ssf + 1024, b[4], b[5], b[6], b[7]);
        const uint32_t tsf = tmem + (quarter * 32u << 16) + kSfCol0 + 16u * stage;
        tmem_st_32x32b_x4(tsf, a0, a1, a2, a3);
        tmem_st_32x32b_x8(tsf + 8, b);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(sf_ready0 + 8u * stage);
        if (++stage == kPStages) stage = 0, phase ^= 1u;
      }
    }
    if (!ok && lane == 0) abort_both();
  } else if (warp == kZeroWarp) {
    // ------------------------ this CTA's rows of the tiles of experts without tokens
    uint8_t* out = static_cast<uint8_t*>(args.out);
    const size_t pitch = static_cast<size_t>(K) * 2;
    const uint64_t zpol = l2_policy_evict_first();
    ItemIter items{total, npairs, 0, pair};
    long long it = 0;
    while (items.next(it)) {
      const int e = s_order[static_cast<int>(it) / per_expert];
      if (s_off[e + 1] != s_off[e]) continue;
      const int tile = static_cast<int>(it) % per_expert;
      const int np = tile / tiles_k, kt = tile % tiles_k;
      uint8_t* base = out + (static_cast<size_t>(e) * N + np * 256 + 128 * rank) * pitch +
                      static_cast<size_t>(kt) * BN * 2 + lane * 16;
      if (!MGW_DIAG_CHECK(np * 256 + 128 * static_cast<int>(rank) + BM <= N && (kt + 1) * BN <= K,
                          args.status))
        continue;
#pragma unroll 4
      for (int r = 0; r < BM; ++r) st_global_zero16_hint(base + r * pitch, zpol);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const int row = quarter * 32 + static_cast<int>(lane);
    const bool store_leader = (ew == 0 && lane == 0);
    const uint32_t acc_empty_leader = map_to_cta(bar_acc_empty, 0);
    const uint64_t opol = l2_policy_evict_first();  // grad_w is written once, never re-read here
    uint32_t acc_phase = 0;
    ItemIter items{total, npairs, 0, pair};
    long long it = 0;
    while (items.next(it)) {
      const int e = s_order[static_cast<int>(it) / per_expert];
      const int tile = static_cast<int>(it) % per_expert;
      const int np = tile / tiles_k, kt = tile % tiles_k;
      const int cnt = s_off[e + 1] - s_off[e];
      if (cnt == 0) continue;  // written by the zero warp
      uint32_t pk[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) pk[j] = 0u;
      const uint64_t t_wait = MGW_DIAG_NOW();
      if (!*abort_flag) {
        if (mbar_wait(bar_acc_full, acc_phase, abort_flag)) {
          tc_fence_after();
          const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 128u * half;
          // four 32-column quarters, each packed to bf16 as soon as it arrives (keeps the
          // live registers within the 480-thread budget)
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(ta + 32 * h, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[16 * h + j] = pack_bf16x2(r[2 * j], r[2 * j + 1]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(acc_empty_leader);
        } else if (lane == 0) {
          abort_both();
        }
        acc_phase ^= 1u;
      }
      const uint32_t stage_base = sbase + kPOffOut;
      const int orow = e * N + np * 256 + 128 * static_cast<int>(rank);
      const bool in_out = MGW_DIAG_CHECK(np * 256 + 128 * static_cast<int>(rank) + 128 <= N &&
                                             kt * BN + 256 <= K,
                                         store_leader ? args.status : nullptr);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (store_leader) bulk_wait_read0();
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
        if (store_leader && !*abort_flag && in_out) {
          tma_store_2d_hint(&args.tm_out, kt * BN + 64 * b, orow, stage_base, opol);
          bulk_commit();
        }
      }
      if (store_leader) MGW_DIAG_ITEM(wgrad, it, t_wait, MGW_DIAG_NOW());
    }
    if (store_leader) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no pair MMA reads this CTA's shared memory or writes its TMEM any more
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

bool wgrad_uses_pair(int E, int N) { return N % 256 == 0 && E <= kMaxPairExperts; }

cudaError_t launch_grouped_wgrad(const WgradArgs& a, int num_sms, cudaStream_t stream) {
  if (!wgrad_uses_pair(a.E, a.N)) {
    static thread_local uint64_t attr_ctx = 0;
    const cudaError_t err = set_smem_attr_once(reinterpret_cast<const void*>(grouped_wgrad_kernel),
                                               wgrad_smem_bytes(kMaxExperts), &attr_ctx);
    if (err != cudaSuccess) return err;
    const long long total = static_cast<long long>(a.N / BM) * (a.K / BN) * a.E;
    long long grid = num_sms;
    if (grid > total) grid = total;
    if (grid < 1) grid = 1;
    grouped_wgrad_kernel<<<static_cast<unsigned>(grid), kThreads, wgrad_smem_bytes(a.E), stream>>>(a);
    return cudaGetLastError();
  }
  static thread_local uint64_t attr_ctx_pair = 0;
  const cudaError_t err = set_smem_attr_once(reinterpret_cast<const void*>(grouped_wgrad_pair_kernel),
                                             wgrad_pair_smem_bytes(kMaxPairExperts), &attr_ctx_pair);
  if (err != cudaSuccess) return err;
  // One CTA pair per two SMs (both dies have an even SM count), at most one pair per item.
  const long long total = static_cast<long long>(a.N / 256) * (a.K / BN) * a.E;
  long long pairs = num_sms / 2;
  if (pairs > total) pairs = total;
  if (pairs < 1) pairs = 1;
  grouped_wgrad_pair_kernel<<<static_cast<unsigned>(2 * pairs), kPThreads,
                              wgrad_pair_smem_bytes(a.E), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mgw
