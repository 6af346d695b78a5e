// Grouped fp32 data gradient with 3xTF32 tcgen05 MMAs on CTA pairs.
//
//   dx[r, k] = sum_n dy[r, n] * W[e(r), n, k],  e(r): the expert whose row range holds r.
//
// The same product and splits as grouped_dgrad_kernel (dgrad.cu): each fp32 operand x is
// split as hi = tf32(x), lo = x - hi (tf32_split) and the product is
// hi*hi + hi*lo + lo*hi accumulated in fp32 in TMEM (Ootomo & Yokota, "Recovering single
// precision accuracy from Tensor Cores while surpassing the FP32 theoretical peak
// performance", IJHPCA 2022).
//
// Work item = (expert e, 256-row pair tile inside e's row range, BNP = 256-column k tile), owned by
// a pair of CTAs in a (2,1,1) cluster: CTA r holds rows 128r .. 128r+127 of the pair tile (its
// A operand in its own TMEM, its accumulator) and k columns (BNP/2)r .. (BNP/2)r + BNP/2 - 1
// of the B operand; the even CTA issues tcgen05.mma.cta_group::2.kind::tf32 (M=256, N=BNP,
// K=8) with A from TMEM.  Measured on the single-SM kernel, the bound is shared-memory bytes
// per MMA: the raw W tile in by TMA, read and split by the transform, the hi/lo tiles written
// and read three times by the MMAs -- about 224 KB per 32-wide chunk against 128 B/clk.  In
// the pair each SM transforms and reads only its half of B, about 112 KB per chunk.
//
// Data path per 32-wide reduction chunk, per CTA:
//   * its half of W[e] rows n (32 of them) arrives raw by TMA into a three-stage ring;
//   * 16 transform warps split it into hi/lo and write it transposed (K-major,
//     128B-swizzled) into a four-stage ring, and split the CTA's 128 dy rows (loaded into
//     registers one chunk ahead) into hi/lo A operands stored into TMEM with tcgen05.st;
//   * both CTAs' transform warps report to the even CTA's full barrier; its MMA thread issues
//     4 K-steps x 3 MMAs and commits the stage back to both CTAs.
//
// Roles (704 threads per CTA):
//   warps 0-3   epilogue: TMEM lane quarter = warp, 32-column chunks -> fp32 stores of the
//               CTA's rows that belong to the item's expert; then the accumulator is
//               released to the even CTA.
//   warp 4      MMA issuer (even CTA).
//   warps 5-20  transform.
//   warp 21     TMA producer of this CTA's raw W tiles.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace mgw {
namespace {

constexpr int BM = 128;    // rows per CTA (half the MMA's M)
constexpr int BK = 32;     // reduction (out_features) per chunk: one 128-byte row of fp32
constexpr int kStages = 4;
constexpr int kRawStages = 3;
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kXfWarp0 = 5;
constexpr int kXfWarps = 16;
constexpr int kXfThreads = kXfWarps * 32;
constexpr int kACols = BK / (kXfWarps / 4);  // A columns per transform warp: 8
constexpr int kTmaWarp = kXfWarp0 + kXfWarps;
constexpr int kThreads = (kTmaWarp + 1) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol0 = 256;  // A operand slots: stage s hi at 256 + 64s, lo at +32
static_assert(kACol0 + 64 * kStages <= kTmemCols, "TMEM budget");

// Shared-memory layout for a pair tile BNP columns wide (each CTA holds BNP/2 B rows).
template <int BNP>
struct Layout {
  static constexpr int kHalf = BNP / 2;                       // B rows (k) per CTA
  static constexpr int kBTile = kHalf * 128;                  // hi or lo: kHalf rows x 128 B
  static constexpr int kStageBytes = 2 * kBTile;
  static constexpr int kRawBytes = BK * kHalf * 4;            // 32 n x kHalf k fp32
  static constexpr int kOffRaw = kStages * kStageBytes;
  static constexpr int kOffBar = kOffRaw + kRawStages * kRawBytes;
  // full[], empty[], raw_full[], raw_empty[], acc_full, acc_empty, done
  static constexpr int kNumBars = 2 * kStages + 2 * kRawStages + 3;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffTable = kOffMisc + 16;
  static constexpr int kParts = kXfThreads / kHalf;           // threads per B row
  static constexpr int kNgPer = (BK / 4) / kParts;            // groups of 4 n per thread
  static_assert(kXfThreads % kHalf == 0 && (BK / 4) % kParts == 0, "transform split");
  static constexpr size_t smem_bytes(int E) {
    return static_cast<size_t>(kOffTable) + sizeof(int) * (3 * static_cast<size_t>(E) + 3) + 1024;
  }
};
constexpr int kPairN = 256;  // the pair tile's columns (each CTA holds 128 of them)
static_assert(Layout<kPairN>::smem_bytes(kMaxExperts) <= 232448, "shared memory budget");

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T over the CTA pair, kind::tf32 (M = 256: each CTA's
// 128 rows of A in its own TMEM; N split over the two CTAs' shared memory).
__device__ __forceinline__ void mma_tf32_at_pair(uint32_t d, uint32_t a_tmem, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  int never = 0;
  (void)mbar_wait(bar, parity, &never);
}

// Item it -> (expert, pair tile in expert, k tile) via the prefix of pair-tile counts.
struct Item {
  int e, pt, kt;
};
__device__ __forceinline__ Item decode_item(long long it, int tiles_k, const int* s_ptp, int E) {
  const int t = static_cast<int>(it / tiles_k);
  Item r;
  r.kt = static_cast<int>(it % tiles_k);
  int lo = 0, hi = E - 1;  // largest e with s_ptp[e] <= t (a non-empty expert)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_ptp[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  r.e = lo;
  r.pt = t - s_ptp[lo];
  return r;
}

template <int BNP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_dgrad_pair_kernel(const __grid_constant__ DgradArgs args) {
  using L = Layout<BNP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int E = args.E, out_f = args.out_f, in_f = args.in_f;
  int* s_misc = reinterpret_cast<int*>(smem + L::kOffMisc);  // [0] tmem [1] abort [2] flag
  int* s_off = reinterpret_cast<int*>(smem + L::kOffTable);
  int* s_pad = s_off + (E + 1);
  int* s_ptp = s_pad + (E + 1);  // prefix of 256-row pair-tile counts, E+1 entries
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&s_misc[1]);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair MMAs
  const bool leader = rank == 0;

  if (tid == 0) s_misc[1] = 0;
  // Both CTAs read the same offsets, so both return here or neither does.
  if (!load_offsets(args.expert_off, E, args.rows, s_off, s_pad, &s_misc[2], args.status)) return;
  // pair tiles per expert: ceil(count / 256), prefix-summed by warp 0, 32 experts per step
  if (tid < 32) {
    int carry = 0;
    if (lane == 0) s_ptp[0] = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + static_cast<int>(lane);
      int v = (e < E) ? (s_off[e + 1] - s_off[e] + 255) / 256 : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= static_cast<uint32_t>(d)) v += y;
      }
      if (e < E) s_ptp[e + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }

  const uint32_t bar0 = sbase + L::kOffBar;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };                          // even CTA
  auto bar_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto bar_raw_full = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
  auto bar_raw_empty = [&](int s) { return bar0 + 8u * (2 * kStages + kRawStages + s); };
  const uint32_t bar_acc_full = bar0 + 8u * (2 * kStages + 2 * kRawStages);
  const uint32_t bar_acc_empty = bar_acc_full + 8u;                               // even CTA
  const uint32_t bar_done = bar_acc_full + 16u;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full(s), 2 * kXfWarps);
      mbar_init(bar_empty(s), 1);
    }
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(bar_raw_full(s), 1);
      mbar_init(bar_raw_empty(s), kXfWarps);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, 2 * kEpiWarps);
    mbar_init(bar_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&args.tm_w);
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(&s_misc[0]), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(s_misc[0]);
  const uint32_t peer_abort = map_to_cta(smem_u32(&s_misc[1]), rank ^ 1u);
  auto abort_both = [&]() {
    *abort_flag = 1;
    st_cluster_u32(peer_abort, 1u);
    if (args.status) atomicOr(args.status, kDevTimeout);
  };

  const int tiles_k = in_f / BNP;
  const long long total = static_cast<long long>(s_ptp[E]) * tiles_k;
  const int nchunks = out_f / BK;
  const long long first = blockIdx.x >> 1, step = gridDim.x >> 1;

  if (warp == kTmaWarp) {
    // ------------------------------------ this CTA's half of the raw W tiles by TMA
    if (lane == 0) {
      int rs = 0;
      uint32_t rph = 0;
      int pending[kRawStages];
      uint32_t pending_phase[kRawStages];
      for (int s = 0; s < kRawStages; ++s) pending[s] = 0, pending_phase[s] = 0;
      bool ok = true;
      for (long long it = first; it < total && ok; it += step) {
        const Item item = decode_item(it, tiles_k, s_ptp, E);
        const int k0 = item.kt * BNP + L::kHalf * static_cast<int>(rank);
        for (int c = 0; c < nchunks; ++c) {
          if (!mbar_wait(bar_raw_empty(rs), rph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_raw_full(rs);
          mbar_arrive_expect_tx(fb, L::kRawBytes);
          tma_load_2d(sbase + L::kOffRaw + rs * L::kRawBytes, &args.tm_w, k0,
                      item.e * out_f + c * BK, fb);
          pending[rs] = 1;
          pending_phase[rs] = rph;
          if (++rs == kRawStages) rs = 0, rph ^= 1u;
        }
      }
      if (!ok) abort_both();
      for (int s = 0; s < kRawStages; ++s)
        if (pending[s]) mbar_wait_drain(bar_raw_full(s), pending_phase[s]);
    }
  } else if (warp >= kXfWarp0) {
    // ----------------------------------------------------------- transform
    const int xw = warp - kXfWarp0;              // 0..15
    const int xt = tid - kXfWarp0 * 32;          // 0..511
    const int bk = xt % L::kHalf;                // the B row k of this thread
    const int ng0 = (xt / L::kHalf) * L::kNgPer; // its first group of 4 reduction elements
    const uint32_t q = static_cast<uint32_t>(warp & 3);  // TMEM lane quarter for A
    const int kh = xw >> 2;                      // A columns 8*kh .. 8*kh+7 of the chunk
    const uint32_t full0 = map_to_cta(bar_full(0), 0);
    int stage = 0, rs = 0;
    uint32_t phase = 0, rph = 0;
    bool ok = true;
    for (long long it = first; it < total && ok; it += step) {
      const Item item = decode_item(it, tiles_k, s_ptp, E);
      const int row0 = s_off[item.e] + item.pt * 2 * BM + BM * static_cast<int>(rank);
      const int valid = min(BM, s_off[item.e + 1] - row0);  // may be <= 0 for the odd CTA
      const int r = static_cast<int>(q) * 32 + static_cast<int>(lane);  // this thread's A row
      const float* dyrow = args.dy + static_cast<size_t>(r < valid ? row0 + r : 0) * out_f + kACols * kh;
      // A: 8 consecutive reduction elements of row r, one chunk ahead of their use
      float4 nxt[kACols / 4];
#pragma unroll
      for (int j = 0; j < kACols / 4; ++j) {
        nxt[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < valid) nxt[j] = __ldg(reinterpret_cast<const float4*>(dyrow) + j);
      }
      for (int c = 0; c < nchunks; ++c) {
        float4 a4[kACols / 4];
#pragma unroll
        for (int j = 0; j < kACols / 4; ++j) {
          a4[j] = nxt[j];
          nxt[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (r < valid && c + 1 < nchunks)
            nxt[j] = __ldg(reinterpret_cast<const float4*>(dyrow + (c + 1) * BK) + j);
        }
        if (!mbar_wait(bar_raw_full(rs), rph, abort_flag) ||
            !mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // B: row k = bk of this CTA's K-major half tile holds W[n][k] for the chunk's 32 n;
        // this thread reads its part of column k of the raw [32 n][kHalf k] tile
        // (conflict-free) and writes 4 x 16 bytes of the hi and lo rows per group of 4 n
        const float* raw = reinterpret_cast<const float*>(smem + L::kOffRaw + rs * L::kRawBytes);
        const uint32_t s_bhi = sbase + stage * L::kStageBytes;
        const uint32_t s_blo = s_bhi + L::kBTile;
#pragma unroll
        for (int g = 0; g < L::kNgPer; ++g) {
          const int ng = ng0 + g;
          uint32_t h[4], l[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) tf32_split(raw[(4 * ng + j) * L::kHalf + bk], h[j], l[j]);
          const uint32_t off = bk * 128 + ((ng ^ (bk & 7)) << 4);
          st_shared_u4(s_bhi + off, h[0], h[1], h[2], h[3]);
          st_shared_u4(s_blo + off, l[0], l[1], l[2], l[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_raw_empty(rs));
        if (++rs == kRawStages) rs = 0, rph ^= 1u;
        // A hi/lo into this stage's TMEM slot, this warp's lane quarter and 8-column group
        {
          uint32_t ah[kACols], al[kACols];
#pragma unroll
          for (int j = 0; j < kACols / 4; ++j) {
            tf32_split(a4[j].x, ah[4 * j], al[4 * j]);
            tf32_split(a4[j].y, ah[4 * j + 1], al[4 * j + 1]);
            tf32_split(a4[j].z, ah[4 * j + 2], al[4 * j + 2]);
            tf32_split(a4[j].w, ah[4 * j + 3], al[4 * j + 3]);
          }
          const uint32_t ta = tmem + (q * 32u << 16) + kACol0 + 64u * stage + kACols * kh;
          tmem_st_x8(ta, ah);
          tmem_st_x8(ta + 32, al);
          tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(full0 + 8u * stage);
        if (++stage == kStages) stage = 0, phase ^= 1u;
      }
    }
    if (!ok && lane == 0) abort_both();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------- MMA issuer (even CTA only)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      constexpr uint16_t kBoth = 0x3;
      constexpr uint32_t idesc = idesc_tf32(2 * BM, BNP);
      const uint64_t b_desc0 = sdesc_kmajor_sw128(sbase);
      for (long long it = first; it < total && ok; it += step) {
        if (!mbar_wait_spin(bar_acc_empty, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        acc_phase ^= 1u;
        tc_fence_after();
        for (int c = 0; c < nchunks; ++c) {
          if (!mbar_wait_spin(bar_full(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bhi = b_desc0 + static_cast<uint32_t>(stage * (L::kStageBytes >> 4));
          const uint64_t blo = bhi + (L::kBTile >> 4);
          const uint32_t ahi = tmem + kACol0 + 64u * stage;
          const uint32_t alo = ahi + 32u;
#pragma unroll
          for (int ks = 0; ks < BK / 8; ++ks) {
            mma_tf32_at_pair(tmem, alo + 8u * ks, bhi + 2 * ks, idesc, (c | ks) != 0);
            mma_tf32_at_pair(tmem, ahi + 8u * ks, blo + 2 * ks, idesc, 1u);
            mma_tf32_at_pair(tmem, ahi + 8u * ks, bhi + 2 * ks, idesc, 1u);
          }
          mma_commit_pair(bar_empty(stage), kBoth);
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit_pair(bar_acc_full, kBoth);
      }
      if (!ok) abort_both();
      mma_commit_pair(bar_done, 0x1);
      mbar_wait_drain(bar_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp;  // warps 0-3
    const uint32_t acc_empty0 = map_to_cta(bar_acc_empty, 0);
    uint32_t acc_phase = 0;
    for (long long it = first; it < total; it += step) {
      if (*abort_flag) break;
      if (!mbar_wait(bar_acc_full, acc_phase, abort_flag)) {
        if (lane == 0) abort_both();
        break;
      }
      acc_phase ^= 1u;
      tc_fence_after();
      const Item item = decode_item(it, tiles_k, s_ptp, E);
      const int row0 = s_off[item.e] + item.pt * 2 * BM + BM * static_cast<int>(rank);
      const int valid = min(BM, s_off[item.e + 1] - row0);
      const int r = quarter * 32 + static_cast<int>(lane);
      float* dst = args.dx + static_cast<size_t>(r < valid ? row0 + r : 0) * in_f + item.kt * BNP;
      const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int j = 0; j < BNP / 32; ++j) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(ta + 32u * j, v);
        tmem_wait_ld();
        if (r < valid) {
#pragma unroll
          for (int qq = 0; qq < 8; ++qq)
            *reinterpret_cast<float4*>(dst + 32 * j + 4 * qq) =
                make_float4(__uint_as_float(v[4 * qq]), __uint_as_float(v[4 * qq + 1]),
                            __uint_as_float(v[4 * qq + 2]), __uint_as_float(v[4 * qq + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(acc_empty0);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no pair MMA reads this CTA's shared memory or TMEM any more
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

bool dgrad_uses_pair(const DgradArgs& a, int num_sms) {
  // Pair tiles of 256 columns when there are at least four rounds of them for the SM pairs
  // (an upper bound of the count: the rows' pair tiles plus one partial per expert).
  // Measured on GB300: the MoE FFN pair (65536 rows, 1536 -> 4096, 64 experts) 3.60 ms on
  // the single-SM kernel, 2.95 ms on pairs; 4096 rows 1024 -> 1024 over 8 experts (80 pair
  // tiles of 256 columns, 160 of 128) stays on the single-SM kernel: 55 us against 89 us for
  // 128-column pair tiles, whose 768 MMA cycles per chunk do not cover the A transform.
  const long long tiles256 = (static_cast<long long>(a.rows) / 256 + a.E) * (a.in_f / 256);
  return a.in_f % 256 == 0 && tiles256 >= 4ll * (num_sms / 2);
}

cudaError_t launch_grouped_dgrad_pair(const DgradArgs& a, int num_sms, cudaStream_t stream) {
  static thread_local uint64_t attr_ctx = 0;
  cudaError_t err = set_smem_attr_once(reinterpret_cast<const void*>(grouped_dgrad_pair_kernel<kPairN>),
                                       Layout<kPairN>::smem_bytes(kMaxExperts), &attr_ctx);
  if (err != cudaSuccess) return err;
  // Upper bound of the item count without reading expert_off on the host.
  const long long max_items = (static_cast<long long>(a.rows) / 256 + a.E) * (a.in_f / kPairN);
  long long pairs = num_sms / 2;
  if (pairs > max_items) pairs = max_items;
  if (pairs < 1) pairs = 1;
  grouped_dgrad_pair_kernel<kPairN><<<static_cast<unsigned>(2 * pairs), kThreads,
                                      Layout<kPairN>::smem_bytes(a.E), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mgw
