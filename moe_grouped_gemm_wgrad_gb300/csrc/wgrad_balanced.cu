// Grouped MXFP8 expert weight gradient, load-balanced for skewed routing:
//
//   grad_w[e*N + n, k] = sum_{t in expert e} g[t, n] * x[t, k]
//
// The same tcgen05 pipeline as the static kernel (TMA producer warp, one MMA-issuing
// thread, 4-stage ring, scale atoms copied to TMEM one chunk ahead, 128x256 fp32
// accumulator drained by eight epilogue warps), with two differences for routings where a
// few experts hold most tokens:
//
// * Split-K over tokens.  An expert whose 128-token chunk count exceeds a target item
//   length L gets S = ceil(chunks / L) parts (at most 16) per output tile; part p covers
//   chunks [p*chunks/S, (p+1)*chunks/S).  L starts at max(8, all chunks / (2 * grid)) so
//   there are about two items per CTA, and doubles until the split tiles' fp32 partials fit
//   the caller's workspace.  Every part writes its 128x256 fp32 partial to its workspace slot,
//   fences, and counts itself on the tile's counter; the part that counts last adds the S
//   partials in part order (its own from registers), so the result does not depend on which
//   part finished last, writes bf16 and resets the counter.  No CTA waits for another.
// * Dynamic scheduling.  Items (expert, tile, part) are ordered by descending part length
//   and handed out by an atomic counter in the workspace, one item ahead, so every CTA takes
//   the next longest item when it is free (greedy LPT).  The producer decodes each item and
//   publishes it through a two-slot shared-memory ring to the MMA thread and the epilogue.  The last CTA
//   to finish resets the counter, leaving the workspace zero-filled for the next call.
//
// Tiles of experts without tokens are written with zeros by a dedicated warp (static
// round-robin over the CTAs), as in the static kernel.
#include <cuda_bf16.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace mgw {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BT = 128;
constexpr int kStages = 4;
constexpr int kABytes = BM * BT;
constexpr int kBBytes = BN * BT;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSfStage = 512 + 1024;
constexpr int kOutBytes = BM * 64 * 2;
constexpr int kItemSlots = 2;
constexpr int kOffOut = kStages * kStageBytes;
constexpr int kOffSf = kOffOut + kOutBytes;
constexpr int kOffBar = kOffSf + kStages * kSfStage;
// full[], empty[], acc_full, acc_empty, done, item_full[], item_empty[]
constexpr int kNumBars = 2 * kStages + 3 + 2 * kItemSlots;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffRing = kOffMisc + 16;
constexpr int kOffTable = kOffRing + kItemSlots * 8 * 4;
constexpr int kThreads = 352;
constexpr int kEpiWarps = 8;
constexpr int kZeroWarp = 10;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;
constexpr int kMaxSplit = 16;
constexpr int kSlotFloats = BM * BN;  // one fp32 partial tile

// Tables: expert_off, padded starts, item prefix by rank, slot base (int, E+1 each),
// order (uint16, E), split factor (uint8, E).
__host__ __device__ constexpr size_t balanced_smem_bytes(int E) {
  return static_cast<size_t>(kOffTable) + sizeof(int) * 4 * (static_cast<size_t>(E) + 1) +
         (sizeof(uint16_t) + 1) * static_cast<size_t>(E) + 1024;
}
static_assert(balanced_smem_bytes(kMaxBalancedExperts) <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void st_cg_v4(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.cg.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

__device__ __forceinline__ float4 ld_cg_v4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  int never = 0;
  (void)mbar_wait(bar, parity, &never);
}

__device__ __forceinline__ long long warp_sum(long long v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Split factor of an expert with `ch` chunks for target item length L.
__device__ __forceinline__ int split_of(int ch, long long L) {
  if (ch <= L) return 1;
  const long long s = (ch + L - 1) / L;
  return static_cast<int>(min(static_cast<long long>(min(kMaxSplit, ch)), s));
}

struct Item {
  int e, nt, kt, tile, part, S, c0, c1;
};

__device__ __forceinline__ Item decode_item(int it, int E, int tiles, int tiles_k, const int* s_off,
                                            const int* s_ipref, const uint16_t* s_order,
                                            const uint8_t* s_split) {
  int lo = 0, hi = E - 1;  // the largest rank whose first item is <= it
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_ipref[mid] <= it)
      lo = mid;
    else
      hi = mid - 1;
  }
  Item x;
  x.e = s_order[lo];
  x.S = s_split[x.e];
  const int local = it - s_ipref[lo];
  x.part = local / tiles;
  x.tile = local % tiles;
  x.nt = x.tile / tiles_k;
  x.kt = x.tile % tiles_k;
  const int ch = (s_off[x.e + 1] - s_off[x.e] + BT - 1) / BT;
  x.c0 = x.part * ch / x.S;  // part <= 16 and ch < 2^24: no overflow
  x.c1 = (x.part + 1) * ch / x.S;
  return x;
}

__device__ __forceinline__ void ring_put(volatile int* slot, const Item& x) {
  slot[0] = x.e, slot[1] = x.nt, slot[2] = x.kt, slot[3] = x.tile;
  slot[4] = x.part, slot[5] = x.S, slot[6] = x.c0, slot[7] = x.c1;
}
__device__ __forceinline__ Item ring_get(const volatile int* slot) {
  Item x;
  x.e = slot[0], x.nt = slot[1], x.kt = slot[2], x.tile = slot[3];
  x.part = slot[4], x.S = slot[5], x.c0 = slot[6], x.c1 = slot[7];
  return x;
}

__global__ void __launch_bounds__(kThreads, 1) grouped_wgrad_balanced_kernel(const __grid_constant__ WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int E = args.E, N = args.N, K = args.K;
  // misc: [0] tmem base [1] abort [2] flag [3] last-part flag; then the item ring: per slot
  // the decoded item (e, nt, kt, tile, part, S, c0, c1), e = -1 after the last item
  int* s_misc = reinterpret_cast<int*>(smem + kOffMisc);
  volatile int* s_ring = reinterpret_cast<volatile int*>(smem + kOffRing);
  int* s_off = reinterpret_cast<int*>(smem + kOffTable);
  int* s_pad = s_off + (E + 1);
  int* s_ipref = s_pad + (E + 1);
  int* s_sbase = s_ipref + (E + 1);
  uint16_t* s_order = reinterpret_cast<uint16_t*>(s_sbase + (E + 1));
  uint8_t* s_split = reinterpret_cast<uint8_t*>(s_order + E);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&s_misc[1]);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane = lane_id();

  if (tid == 0) s_misc[1] = 0;
  if (!load_offsets(args.expert_off, E, args.M, s_off, s_pad, &s_misc[2], args.status)) return;

  const int tiles_n = N / BM, tiles_k = K / BN;
  const int tiles = tiles_n * tiles_k;
  auto chunks = [&](int e) { return (s_off[e + 1] - s_off[e] + BT - 1) / BT; };

  // ---- split factors: every CTA makes the same choice
  if (warp == 0) {
    long long tot = 0;
    for (int e = static_cast<int>(lane); e < E; e += 32) tot += chunks(e);
    tot = warp_sum(tot) * tiles;
    long long L = (tot + 2ll * gridDim.x - 1) / (2ll * gridDim.x);
    if (L < 8) L = 8;
    for (int iter = 0; iter < 48; ++iter) {
      long long slots = 0;
      for (int e = static_cast<int>(lane); e < E; e += 32) {
        const int s = split_of(chunks(e), L);
        if (s > 1) slots += static_cast<long long>(tiles) * s;
      }
      if (warp_sum(slots) <= args.ws_slots) break;
      L *= 2;
    }
    for (int e = static_cast<int>(lane); e < E; e += 32) {
      int s = split_of(chunks(e), L);
      if (args.ws_slots <= 0) s = 1;
      s_split[e] = static_cast<uint8_t>(s);
    }
  }
  __syncthreads();
  // ---- order: descending part length (experts without tokens last), ties by index
  for (int e = tid; e < E; e += kThreads) {
    const int ce = chunks(e);
    const int ke = ce > 0 ? (ce + s_split[e] - 1) / s_split[e] : 0;
    int rank = 0;
    for (int j = 0; j < E; ++j) {
      const int cj = chunks(j);
      const int kj = cj > 0 ? (cj + s_split[j] - 1) / s_split[j] : 0;
      rank += (kj > ke) || (kj == ke && j < e);
    }
    s_order[rank] = static_cast<uint16_t>(e);
  }
  __syncthreads();
  // ---- item prefix by rank and partial-slot base by expert (warp 0, 32 at a time)
  if (warp == 0) {
    int carry_i = 0, carry_s = 0;
    if (lane == 0) s_ipref[0] = 0, s_sbase[0] = 0;
    for (int base = 0; base < E; base += 32) {
      const int i = base + static_cast<int>(lane);
      int vi = 0, vs = 0;
      if (i < E) {
        const int er = s_order[i];
        vi = chunks(er) > 0 ? tiles * s_split[er] : 0;
        vs = s_split[i] > 1 ? tiles * s_split[i] : 0;
      }
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int yi = __shfl_up_sync(0xffffffffu, vi, d);
        const int ys = __shfl_up_sync(0xffffffffu, vs, d);
        if (lane >= static_cast<uint32_t>(d)) vi += yi, vs += ys;
      }
      if (i < E) s_ipref[i + 1] = carry_i + vi, s_sbase[i + 1] = carry_s + vs;
      carry_i += __shfl_sync(0xffffffffu, vi, 31);
      carry_s += __shfl_sync(0xffffffffu, vs, 31);
    }
  }

  const uint32_t bar0 = sbase + kOffBar;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t bar_acc_full = bar0 + 8u * (2 * kStages);
  const uint32_t bar_acc_empty = bar0 + 8u * (2 * kStages + 1);
  const uint32_t bar_done = bar0 + 8u * (2 * kStages + 2);
  auto bar_item_full = [&](int s) { return bar0 + 8u * (2 * kStages + 3 + s); };
  auto bar_item_empty = [&](int s) { return bar0 + 8u * (2 * kStages + 3 + kItemSlots + s); };
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, kEpiWarps);
    mbar_init(bar_done, 1);
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(bar_item_full(s), 1);
      mbar_init(bar_item_empty(s), 1 + kEpiWarps);  // the MMA thread and each epilogue warp
    }
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
  const int total_items = s_ipref[E];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int pending[kStages];
      uint32_t pending_phase[kStages];
      for (int s = 0; s < kStages; ++s) pending[s] = 0, pending_phase[s] = 0;
      bool ok = true;
      int islot = 0;
      uint32_t iph = 0;
      int nxt = atomicAdd(&args.ws_sched[0], 1);
      while (ok) {
        const int it = nxt;
        const bool have = it < total_items;
        if (have) nxt = atomicAdd(&args.ws_sched[0], 1);  // one item ahead
        if (!mbar_wait(bar_item_empty(islot), iph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        Item x{-1, 0, 0, 0, 0, 1, 0, 0};
        if (have) x = decode_item(it, E, tiles, tiles_k, s_off, s_ipref, s_order, s_split);
        ring_put(s_ring + 8 * islot, x);
        mbar_arrive(bar_item_full(islot));
        if (++islot == kItemSlots) islot = 0, iph ^= 1u;
        if (!have) break;
        const int ch0 = s_pad[x.e] / BT;
        for (int c = x.c0; c < x.c1; ++c) {
          if (!mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full(stage);
          mbar_arrive_expect_tx(fb, kStageBytes + kSfStage);
          const uint32_t sa = sbase + stage * kStageBytes;
          const int tok = (ch0 + c) * BT;
          tma_load_2d(sa, &args.tm_a, tok, x.nt * BM, fb);
          tma_load_2d(sa + kABytes, &args.tm_b, tok, x.kt * BN, fb);
          const uint32_t ssf = sbase + kOffSf + stage * kSfStage;
          bulk_load(ssf, args.gs + (static_cast<size_t>(ch0 + c) * tiles_n + x.nt) * 512, 512, fb);
          bulk_load(ssf + 512,
                    args.xs + (static_cast<size_t>(ch0 + c) * (K / 128) + 2 * x.kt) * 512, 1024, fb);
          pending[stage] = 1;
          pending_phase[stage] = phase;
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        if (args.status) atomicOr(args.status, kDevTimeout);
      }
      for (int s = 0; s < kStages; ++s)
        if (pending[s]) mbar_wait_drain(bar_full(s), pending_phase[s]);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      int islot = 0;
      uint32_t iph = 0;
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
      while (ok) {
        if (!mbar_wait(bar_item_full(islot), iph, abort_flag)) {
          ok = false;
          break;
        }
        const Item x = ring_get(s_ring + 8 * islot);
        mbar_arrive(bar_item_empty(islot));
        if (++islot == kItemSlots) islot = 0, iph ^= 1u;
        if (x.e < 0) break;
        const int cnt = s_off[x.e + 1] - s_off[x.e];
        if (!stage_scales(stage, phase) || !mbar_wait(bar_acc_empty, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int full_chunks = cnt / BT;
        for (int c = x.c0; c < x.c1; ++c) {
          const uint32_t tsf = tmem + kSfCol0 + 16u * stage;
          const uint64_t ad = a_desc0 + static_cast<uint32_t>(stage * (kStageBytes >> 4));
          const uint64_t bd = ad + (kABytes >> 4);
          if (c < full_chunks) {
            mma_mxf8_chunk128<BM, BN>(tmem, ad, bd, tsf, tsf + 8, c != x.c0 ? 1u : 0u);
          } else {
            const int nkb = (cnt - c * BT + 31) / 32;
            for (int kb = 0; kb < nkb; ++kb) {
              mma_mxf8_block32(tmem, ad + 2 * kb, bd + 2 * kb, idesc_mxf8_e4m3(BM, BN, kb, kb),
                               tsf, tsf + 8, (c != x.c0 || kb != 0) ? 1u : 0u);
            }
          }
          // release the stage as soon as its MMAs are issued, then prepare the next one
          mma_commit(bar_empty(stage));
          if (++stage == kStages) stage = 0, phase ^= 1u;
          if (c + 1 < x.c1 && !stage_scales(stage, phase)) {
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
  } else if (warp == kZeroWarp) {
    // ----------------------------------- zero tiles of experts without tokens (static)
    uint8_t* out = static_cast<uint8_t*>(args.out);
    const size_t pitch = static_cast<size_t>(K) * 2;
    const long long grid = gridDim.x;
    long long zbase = 0;  // zero tiles before expert e; tile z goes to CTA z % grid
    for (int e = 0; e < E; ++e) {
      if (s_off[e + 1] != s_off[e]) continue;
      const long long first = ((static_cast<long long>(blockIdx.x) - zbase) % grid + grid) % grid;
      zbase += tiles;
      for (long long tile = first; tile < tiles; tile += grid) {
        const int nt = static_cast<int>(tile) / tiles_k, kt = static_cast<int>(tile) % tiles_k;
        uint8_t* base = out + (static_cast<size_t>(e) * N + nt * BM) * pitch +
                        static_cast<size_t>(kt) * BN * 2 + lane * 16;
#pragma unroll 4
        for (int r = 0; r < BM; ++r)
          *reinterpret_cast<uint4*>(base + r * pitch) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const int row = quarter * 32 + static_cast<int>(lane);
    const bool leader = (ew == 0 && lane == 0);
    volatile int* s_last = reinterpret_cast<volatile int*>(&s_misc[3]);
    uint32_t acc_phase = 0;
    int islot = 0;
    uint32_t iph = 0;
    while (true) {
      if (!mbar_wait(bar_item_full(islot), iph, abort_flag)) {
        *abort_flag = 1;
        if (lane == 0 && args.status) atomicOr(args.status, kDevTimeout);
        break;
      }
      const Item x = ring_get(s_ring + 8 * islot);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_item_empty(islot));
      if (++islot == kItemSlots) islot = 0, iph ^= 1u;
      if (x.e < 0) break;
      uint32_t r[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) r[j] = 0u;
      bool have = false;
      if (!*abort_flag) {
        if (mbar_wait(bar_acc_full, acc_phase, abort_flag)) {
          tc_fence_after();
          const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 128u * half;
          tmem_ld_32x32b_x32(ta + 0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          tmem_ld_32x32b_x32(ta + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          tmem_ld_32x32b_x32(ta + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
          tmem_ld_32x32b_x32(ta + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acc_empty);
          have = true;
        } else {
          *abort_flag = 1;
          if (lane == 0 && args.status) atomicOr(args.status, kDevTimeout);
        }
        acc_phase ^= 1u;
      }
      uint32_t pk[64];
      bool store = true;
      if (x.S == 1) {
#pragma unroll
        for (int j = 0; j < 64; ++j) pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
      } else {
        // fp32 partial of this part; float4 j4 of this thread's row at
        // ((half * 32 + j4) * 128 + row) * 4 floats, so a warp writes 512 contiguous bytes
        const int slot0 = s_sbase[x.e] + x.tile;          // part 0's slot: the tile counter
        const int tile_parts = tiles;                       // slot stride between parts
        float* own = args.ws_part + static_cast<size_t>(slot0 + x.part * tile_parts) * kSlotFloats;
        if (have) {
#pragma unroll
          for (int j4 = 0; j4 < 32; ++j4)
            st_cg_v4(own + ((half * 32 + j4) * 128 + row) * 4, __uint_as_float(r[4 * j4]),
                     __uint_as_float(r[4 * j4 + 1]), __uint_as_float(r[4 * j4 + 2]),
                     __uint_as_float(r[4 * j4 + 3]));
        }
        __threadfence();
        named_bar_sync(2, kEpiWarps * 32);
        if (leader) *s_last = (atomicAdd(&args.ws_cnt[slot0], 1) == x.S - 1) ? 1 : 0;
        named_bar_sync(2, kEpiWarps * 32);
        store = *s_last != 0;
        if (store) {
          __threadfence();
          // sum of the S partials in part order; this part's from registers
#pragma unroll
          for (int j4 = 0; j4 < 32; ++j4) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            for (int p = 0; p < x.S; ++p) {
              float4 v;
              if (p == x.part) {
                v = make_float4(__uint_as_float(r[4 * j4]), __uint_as_float(r[4 * j4 + 1]),
                                __uint_as_float(r[4 * j4 + 2]), __uint_as_float(r[4 * j4 + 3]));
              } else {
                v = ld_cg_v4(args.ws_part + static_cast<size_t>(slot0 + p * tile_parts) * kSlotFloats +
                             ((half * 32 + j4) * 128 + row) * 4);
              }
              if (p == 0) {
                a0 = v.x, a1 = v.y, a2 = v.z, a3 = v.w;
              } else {
                a0 += v.x, a1 += v.y, a2 += v.z, a3 += v.w;
              }
            }
            pk[2 * j4] = pack_bf16x2(a0, a1);
            pk[2 * j4 + 1] = pack_bf16x2(a2, a3);
          }
          if (leader) atomicExch(&args.ws_cnt[slot0], 0);  // zero again for the next call
        }
      }
      if (!store) continue;
      const uint32_t stage_base = sbase + kOffOut;
      const int orow = x.e * N + x.nt * BM;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (leader) bulk_wait_read0();
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
          tma_store_2d(&args.tm_out, x.kt * BN + 64 * b, orow, stage_base);
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
  // The last CTA to finish zeroes the item counter for the next call (every CTA has
  // fetched its last item before its final barrier above).
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&args.ws_sched[1], 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(&args.ws_sched[0], 0);
      atomicExch(&args.ws_sched[1], 0);
    }
  }
}

}  // namespace

int balanced_workspace_slots(size_t bytes) {
  if (bytes < kWsHeaderBytes) return -1;
  long long s = static_cast<long long>((bytes - kWsHeaderBytes) / (static_cast<size_t>(kSlotFloats) * 4 + 4));
  while (s > 0 && kWsHeaderBytes + ((4 * static_cast<size_t>(s) + 255) & ~size_t(255)) +
                          static_cast<size_t>(s) * kSlotFloats * 4 > bytes)
    --s;
  if (s > (1 << 24)) s = 1 << 24;
  return static_cast<int>(s);
}

size_t balanced_workspace_bytes(int slots) {
  return kWsHeaderBytes + ((4 * static_cast<size_t>(slots) + 255) & ~size_t(255)) +
         static_cast<size_t>(slots) * kSlotFloats * 4;
}

cudaError_t launch_grouped_wgrad_balanced(WgradArgs a, void* workspace, int slots, int num_sms,
                                          cudaStream_t stream) {
  static thread_local uint64_t attr_ctx = 0;
  cudaError_t err = set_smem_attr_once(
      reinterpret_cast<const void*>(grouped_wgrad_balanced_kernel),
      balanced_smem_bytes(kMaxBalancedExperts), &attr_ctx);
  if (err != cudaSuccess) return err;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.ws_sched = reinterpret_cast<int*>(ws);
  a.ws_cnt = reinterpret_cast<int*>(ws + kWsHeaderBytes);
  a.ws_part = reinterpret_cast<float*>(ws + kWsHeaderBytes + ((4 * static_cast<size_t>(slots) + 255) & ~size_t(255)));
  a.ws_slots = slots;
  // One CTA per SM: split items can outnumber the output tiles.
  const long long grid = num_sms > 0 ? num_sms : 1;
  grouped_wgrad_balanced_kernel<<<static_cast<unsigned>(grid), kThreads, balanced_smem_bytes(a.E), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mgw
