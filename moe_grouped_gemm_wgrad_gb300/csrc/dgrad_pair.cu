// Grouped fp32 data gradient with 3xTF32 tcgen05 MMAs on CTA pairs.
//
//   dx[r, k] = sum_n dy[r, n] * W[e(r), n, k],  e(r): the expert whose row range holds r.
//
// The product, the operand splits and the staging are those of the single-SM kernel
// (dgrad.cuh).  Work item = (expert e, 256-row pair tile inside e's row range, 256-column k
// tile), owned by a pair of CTAs in a (2,1,1) cluster: CTA r holds rows 128r .. 128r+127 of
// the pair tile (its A operand in its own TMEM, its accumulator) and k columns
// 128r .. 128r+127 of the B operand; the even CTA issues tcgen05.mma.cta_group::2.kind::tf32
// (M=256, N=256, K=8).  Each SM transforms and reads only its half of B, so per 16-wide half
// chunk a CTA moves about 72 KB through shared memory (W and dy in by TMA and read once, 16 KB
// of hi|lo B written, 24 KB read by the MMAs) against 768 MMA cycles: the MMAs, not shared
// memory, bound it, where the single-SM kernel moves ~128 KB per 768 cycles.  It is used when
// there are enough 256-row pair tiles to keep the SM pairs busy.
//
// Roles (672 threads per CTA):
//   warps 0-3   epilogue: TMEM lane quarter = warp, the CTA's rows that belong to the item's
//               expert.  Lane 0 of warp 0 of the even CTA issues each item's MMAs before its
//               share of the epilogue (one accumulator: the next item's MMAs wait for both
//               CTAs' epilogues anyway).
//   warps 4-19  transform: per half chunk, thread t writes 4 reduction elements of B row
//               t % 128 and splits 4 A elements of one row (four warps per TMEM lane
//               quarter, 4 columns each); both CTAs report to the even CTA's full barrier.
//   warp 20     TMA producer of this CTA's raw W and dy tiles, which also prefetches the next
//               eight chunks of both into L2.
#include <cstdint>

#include "dgrad.cuh"

namespace mgw {

MGW_DIAG_TIMELINE_DEFINE(dgrad_pair, 3)

namespace {

using namespace dgrad;

constexpr int BM = 128;         // rows per CTA (half the MMA's M)
constexpr int BNP = 256;        // dx columns per pair tile (MMA N)
constexpr int kHalfN = BNP / 2; // B rows (k) per CTA
constexpr int kStages = 4;
constexpr int kRawStages = 4;
constexpr int kPrefetch = 8;    // chunks of W and dy prefetched into L2 ahead of the TMA loads
constexpr int kStageBytes = kHalfN * 128;        // 128 B rows of 16 hi | 16 lo tf32: 16 KB
constexpr int kRawW = BK * kHalfN * 4;           // raw W rows: 32 n x 128 k fp32 = 16 KB
constexpr int kRawBytes = kRawW + kRawDy;        // + 128 dy rows x 32 n = 32 KB
constexpr int kOffRaw = kStages * kStageBytes;   // 64 KB
constexpr int kOffBar = kOffRaw + kRawStages * kRawBytes;  // 192 KB
// full[], empty[], raw_full[], raw_empty[], acc_full, acc_empty, done
constexpr int kNumBars = 2 * kStages + 2 * kRawStages + 3;
constexpr int kOffMisc = kOffBar + ((kNumBars * 8 + 15) & ~15);
constexpr int kOffTable = kOffMisc + 16;
constexpr int kEpiWarps = 4;
constexpr int kXfWarp0 = 4;
constexpr int kXfWarps = 16;
constexpr int kXfThreads = kXfWarps * 32;
constexpr int kTmaWarp = kXfWarp0 + kXfWarps;
constexpr int kThreads = (kTmaWarp + 1) * 32;
constexpr int kBN = BKH / (kXfThreads / kHalfN);  // B elements per thread and half chunk: 4
static_assert(kBN == 4 && BM == kRowsPerCta, "transform split");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol0 = 256;  // A operand slots: stage s hi at 256 + 32s, lo at +16
static_assert(kACol0 + 32 * kStages <= kTmemCols, "TMEM budget");

__host__ __device__ constexpr size_t pair_smem_bytes(int E) {
  return static_cast<size_t>(kOffTable) + sizeof(int) * (3 * static_cast<size_t>(E) + 3) + 1024;
}
static_assert(pair_smem_bytes(kMaxExperts) <= 232448, "shared memory budget");

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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_dgrad_pair_kernel(const __grid_constant__ DgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int E = args.E, out_f = args.out_f, in_f = args.in_f;
  int* s_misc = reinterpret_cast<int*>(smem + kOffMisc);  // [0] tmem [1] abort [2] flag
  int* s_off = reinterpret_cast<int*>(smem + kOffTable);
  int* s_pad = s_off + (E + 1);
  int* s_ptp = s_pad + (E + 1);  // prefix of 256-row pair-tile counts, E+1 entries
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&s_misc[1]);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair MMAs
  const bool leader = rank == 0;

  const uint32_t bar0 = sbase + kOffBar;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };                          // even CTA
  auto bar_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto bar_raw_full = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
  auto bar_raw_empty = [&](int s) { return bar0 + 8u * (2 * kStages + kRawStages + s); };
  const uint32_t bar_acc_full = bar0 + 8u * (2 * kStages + 2 * kRawStages);
  const uint32_t bar_acc_empty = bar_acc_full + 8u;                               // even CTA
  const uint32_t bar_done = bar_acc_full + 16u;
  // Barriers, TMEM and the tensor maps are set up while the offsets are read.
  if (tid == 0) {
    s_misc[1] = 0;
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
    tma_prefetch_desc(&args.tm_dy);
  }
  if (warp == 0) {
    tmem_alloc_pair(smem_u32(&s_misc[0]), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // Both CTAs read the same offsets, so both leave here or neither does.
  const bool offsets_ok = load_offsets(args.expert_off, E, args.rows, s_off, s_pad, &s_misc[2], args.status);
  tc_fence_after();  // load_offsets ends with a block barrier
  const uint32_t tmem = static_cast<uint32_t>(s_misc[0]);
  if (!offsets_ok) {
    cluster_sync();
    if (warp == 0) tmem_dealloc_pair(tmem, kTmemCols);
    return;
  }
  // pair tiles per expert: ceil(count / 256), prefix-summed by warp 0, 32 experts per step
  if (tid < 32) {
    int carry = 0;
    if (lane == 0) s_ptp[0] = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + static_cast<int>(lane);
      int v = (e < E) ? (s_off[e + 1] - s_off[e] + 2 * BM - 1) / (2 * BM) : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= static_cast<uint32_t>(d)) v += y;
      }
      if (e < E) s_ptp[e + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrive
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
    // ------------------------------------ this CTA's raw W and dy tiles by TMA
    if (lane == 0) {
      int rs = 0;
      uint32_t rph = 0;
      int pending[kRawStages];
      uint32_t pending_phase[kRawStages];
      for (int s = 0; s < kRawStages; ++s) pending[s] = 0, pending_phase[s] = 0;
      bool ok = true;
      bool dropped = false;
      const int k_half = kHalfN * static_cast<int>(rank);
      const int r_half = BM * static_cast<int>(rank);
      // L2 prefetch cursor over this pair's (item, chunk) sequence, kPrefetch chunks ahead of
      // the loads; the ring's first loads go out first and the cursor catches up two chunks
      // per load.
      long long pf_it = first;
      int pf_c = 0, pf_row0 = 0;
      Item pf_item{0, 0, 0};
      auto pf_set = [&]() {
        if (pf_it < total) {
          pf_item = decode_item(pf_it, tiles_k, s_ptp, E);
          pf_row0 = s_off[pf_item.e] + pf_item.rt * 2 * BM + r_half;
        }
      };
      auto pf_advance = [&](bool prefetch) {
        if (pf_it >= total) return;
        if (prefetch) {
          tma_prefetch_l2_2d(&args.tm_w, pf_item.kt * BNP + k_half, pf_item.e * out_f + pf_c * BK);
          tma_prefetch_l2_2d(&args.tm_dy, pf_c * BK, pf_row0);
        }
        if (++pf_c == nchunks) {
          pf_c = 0;
          pf_it += step;
          pf_set();
        }
      };
      pf_set();
      for (int i = 0; i < kRawStages; ++i) pf_advance(false);
      int ahead = kRawStages;
      for (long long it = first; it < total && ok; it += step) {
        const Item item = decode_item(it, tiles_k, s_ptp, E);
        const int row0 = s_off[item.e] + item.rt * 2 * BM + r_half;
        for (int c = 0; c < nchunks; ++c) {
          if (!mbar_wait(bar_raw_empty(rs), rph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_raw_full(rs);
          const uint32_t dst = sbase + kOffRaw + rs * kRawBytes;
          mbar_arrive_expect_tx(fb, kRawBytes);
          if (args.drop_first_load && !dropped) {  // test hook: this stage never fills
            dropped = true;
            pending[rs] = 1;
            pending_phase[rs] = rph;
            if (++rs == kRawStages) rs = 0, rph ^= 1u;
            continue;
          }
          (void)MGW_DIAG_CHECK(item.e * out_f + (c + 1) * BK <= E * out_f &&
                                   item.kt * BNP + k_half + kHalfN <= in_f && (c + 1) * BK <= out_f,
                               args.status);
          tma_load_2d(dst, &args.tm_w, item.kt * BNP + k_half, item.e * out_f + c * BK, fb);
          tma_load_2d(dst + kRawW, &args.tm_dy, c * BK, row0, fb);
          --ahead;
          for (int k = 0; k < 2 && ahead < kPrefetch; ++k, ++ahead) pf_advance(true);
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
    const int bk = xt % kHalfN;                  // the B row (k within this CTA's half)
    const int part = xt / kHalfN;                // its 4 of the half chunk's 16 n
    const uint32_t q = static_cast<uint32_t>(warp & 3);  // TMEM lane quarter for A
    const int kh = xw >> 2;                      // A columns 4*kh .. 4*kh+3 of a half chunk
    const uint32_t sw_b = static_cast<uint32_t>(bk & 7);  // 128B swizzle of B row bk
    const uint32_t full0 = map_to_cta(bar_full(0), 0);
    int stage = 0, rs = 0;
    uint32_t phase = 0, rph = 0;
    bool ok = true;
    for (long long it = first; it < total && ok; it += step) {
      for (int c = 0; c < nchunks; ++c) {
        if (!mbar_wait(bar_raw_full(rs), rph, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t raw_w = sbase + kOffRaw + rs * kRawBytes;
        const uint32_t raw_dy = raw_w + kRawW;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // W[n][k] for n = 16h + 4part + j of the chunk: column bk of the raw [32 n][128 k]
          // tile (a warp reads 32 consecutive k: conflict-free)
          float w[kBN];
#pragma unroll
          for (int j = 0; j < kBN; ++j)
            w[j] = ld_shared_f32(raw_w + static_cast<uint32_t>(((BKH * h + kBN * part + j) * kHalfN + bk) * 4));
          const float4 a = load_a(raw_dy, h, q, lane, kh);
          if (!mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // B row bk: hi in 16-byte chunk `part`, lo in chunk 4 + part (logical), 128B-swizzled
          {
            uint32_t hi[kBN], lo[kBN];
#pragma unroll
            for (int j = 0; j < kBN; ++j) tf32_split(w[j], hi[j], lo[j]);
            const uint32_t row = sbase + stage * kStageBytes + bk * 128;
            st_shared_u4(row + ((static_cast<uint32_t>(part) ^ sw_b) << 4), hi[0], hi[1], hi[2], hi[3]);
            st_shared_u4(row + ((static_cast<uint32_t>(part + 4) ^ sw_b) << 4), lo[0], lo[1], lo[2], lo[3]);
          }
          // A hi/lo into this stage's TMEM slot, this warp's lane quarter and 4-column group
          store_a(a, q, kh, tmem, kACol0 + 32u * stage);
          tmem_wait_st();
          fence_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(full0 + 8u * stage);
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        // both halves of the raw stage are read
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_raw_empty(rs));
        if (++rs == kRawStages) rs = 0, rph ^= 1u;
      }
    }
    if (!ok && lane == 0) abort_both();
  } else {
    // ----------------------- MMA issuer (even CTA: warp 0, lane 0) and epilogue (both CTAs)
    const int quarter = warp;  // warps 0-3
    const bool issuer = leader && warp == 0 && lane == 0;
    const uint32_t acc_empty0 = map_to_cta(bar_acc_empty, 0);
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    constexpr uint16_t kBoth = 0x3;
    constexpr uint32_t idesc = idesc_tf32(2 * BM, BNP);
    const uint64_t b_desc0 = sdesc_kmajor_sw128(sbase);
    const int nhalves = 2 * nchunks;
    for (long long it = first; it < total; it += step) {
      if (issuer && ok) {
        // both CTAs' epilogues of the previous item have read their accumulators
        ok = mbar_wait_spin(bar_acc_empty, acc_phase ^ 1u, abort_flag);
        tc_fence_after();
        for (int hc = 0; hc < nhalves && ok; ++hc) {
          if (!mbar_wait_spin(bar_full(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // B row: hi at bytes 0-63 (K-steps at +0, +32), lo at 64-127 (desc units of 16 B)
          const uint64_t bhi = b_desc0 + static_cast<uint32_t>(stage * (kStageBytes >> 4));
          const uint64_t blo = bhi + 4;
          const uint32_t ahi = tmem + kACol0 + 32u * stage;
          const uint32_t alo = ahi + 16u;
#pragma unroll
          for (int ks = 0; ks < BKH / 8; ++ks) {
            mma_tf32_at_pair(tmem, alo + 8u * ks, bhi + 2 * ks, idesc, (hc | ks) != 0);
            mma_tf32_at_pair(tmem, ahi + 8u * ks, blo + 2 * ks, idesc, 1u);
            mma_tf32_at_pair(tmem, ahi + 8u * ks, bhi + 2 * ks, idesc, 1u);
          }
          mma_commit_pair(bar_empty(stage), kBoth);
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
        if (ok)
          mma_commit_pair(bar_acc_full, kBoth);
        else
          abort_both();
      }
      __syncwarp();
      if (*abort_flag) break;
      const uint64_t t_wait = MGW_DIAG_NOW();
      if (!mbar_wait(bar_acc_full, acc_phase, abort_flag)) {
        if (lane == 0) abort_both();
        break;
      }
      acc_phase ^= 1u;
      tc_fence_after();
      const Item item = decode_item(it, tiles_k, s_ptp, E);
      const int row0 = s_off[item.e] + item.rt * 2 * BM + BM * static_cast<int>(rank);
      const int valid = min(BM, s_off[item.e + 1] - row0);  // may be <= 0 for the odd CTA
      store_acc_rows(args, tmem, quarter, lane, row0, valid, item.kt * BNP, BNP);
      if (warp == 0 && lane == 0) MGW_DIAG_ITEM(dgrad_pair, it, t_wait, MGW_DIAG_NOW());
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(acc_empty0);
    }
    if (issuer) {
      mma_commit_pair(bar_done, 0x1);
      mbar_wait_drain(bar_done, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no pair MMA reads this CTA's shared memory or TMEM any more
  tc_fence_after();
  if (warp == 0) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

bool dgrad_uses_pair(const DgradArgs& a, int num_sms) {
  // Pair tiles of 256 rows when there are at least four rounds of them for the SM pairs (an
  // upper bound of the count: the rows' pair tiles plus one partial per expert).  4096 rows
  // over 8 experts (80 pair tiles for 76 SM pairs) stay on the single-SM kernel, whose 144
  // tiles of 128 rows fill the SMs in one round.
  const long long tiles256 = (static_cast<long long>(a.rows) / 256 + a.E) * (a.in_f / 256);
  return a.in_f % 256 == 0 && tiles256 >= 4ll * (num_sms / 2);
}

cudaError_t launch_grouped_dgrad_pair(const DgradArgs& a, int num_sms, cudaStream_t stream) {
  static thread_local uint64_t attr_ctx = 0;
  cudaError_t err = set_smem_attr_once(reinterpret_cast<const void*>(grouped_dgrad_pair_kernel),
                                       pair_smem_bytes(kMaxExperts), &attr_ctx);
  if (err != cudaSuccess) return err;
  // Upper bound of the item count without reading expert_off on the host.
  const long long max_items = (static_cast<long long>(a.rows) / 256 + a.E) * (a.in_f / BNP);
  long long pairs = num_sms / 2;
  if (pairs > max_items) pairs = max_items;
  if (pairs < 1) pairs = 1;
  grouped_dgrad_pair_kernel<<<static_cast<unsigned>(2 * pairs), kThreads, pair_smem_bytes(a.E),
                              stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mgw
