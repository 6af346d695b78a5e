// Grouped fp32 data gradient with 3xTF32 tcgen05 MMAs, one SM per output tile.
//
//   dx[r, k] = sum_n dy[r, n] * W[e(r), n, k],  e(r): the expert whose row range holds r.
//
// Work item = (expert e, 128-row tile inside e's row range, 256-column k tile).
// Tiles start at expert_off[e], so a tile never mixes experts: rows of the tile
// past the expert's last row hold whatever dy holds there (zeros past the last row),
// give accumulator rows that are never stored, and change no stored row.  This replaces
// the dgrad page's split between a tiled path and a per-element path for tiles
// that straddle an expert boundary.
//
// Precision: each fp32 operand x is split as hi = tf32(x), lo = x - hi
// (tf32_split), and the product is hi*hi + hi*lo + lo*hi
// accumulated in fp32 in TMEM (Ootomo & Yokota, "Recovering single precision
// accuracy from Tensor Cores while surpassing the FP32 theoretical peak
// performance", IJHPCA 2022).
//
// Data path per 32-wide reduction chunk:
//   * TMA brings W[e] rows n (32 of them, 256 k columns, 32 KB) and the tile's dy rows
//     (128 rows x 32 n, 16 KB, 128B-swizzled) into a two-stage raw ring;
//   * per 16-wide half of the chunk, the transform warps read W column-wise, split it and
//     write the MMA's B operand transposed (K-major, 128B-swizzled, hi in the first and lo
//     in the second 64 bytes of each row) into a three-stage ring, and read dy row-wise,
//     split it and store the hi/lo A operands into TMEM with tcgen05.st;
//   * the MMA thread issues 2 K-steps x 3 tcgen05.mma.kind::tf32 (M=128, N=256, K=8) per
//     half, A from TMEM and B from shared memory, into one 256-column accumulator.
// Every shared-memory access of the transform is conflict-free and every global read goes
// through TMA: per 16-wide half the L1 data pipe moves about 450 wavefronts against 768
// MMA cycles.  (Reading W and dy with per-thread global loads, or dy rows one per lane,
// made that pipe the bound at ~2150 wavefronts per 32-wide chunk.)
//
// Roles (672 threads):
//   warps 0-3   epilogue: TMEM lane quarter = warp, 32-column chunks -> fp32 stores of
//               the rows that belong to the item's expert, then the accumulator is free.
//               Lane 0 of warp 0 issues each item's MMAs before its share of the epilogue:
//               with one accumulator the next item's MMAs wait for the epilogue anyway.
//   warps 4-19  transform: per half chunk, thread t writes 8 reduction elements of B row
//               t % 256 and splits 4 A elements of one row (four warps per TMEM lane
//               quarter, 4 columns each).
//   warp 20     TMA producer of the raw W and dy tiles, which also prefetches the next eight
//               chunks of both into L2.
#include <cstdint>

#include "dgrad.cuh"

namespace mgw {

MGW_DIAG_TIMELINE_DEFINE(dgrad, 2)

namespace {

using namespace dgrad;

constexpr int BM = 128;   // rows per tile (MMA M)
constexpr int BN = 256;   // dx columns per tile (MMA N)
constexpr int kStages = 3;
constexpr int kRawStages = 2;
constexpr int kPrefetch = 8;    // chunks of W and dy prefetched into L2 ahead of the TMA loads
constexpr int kStageBytes = BN * 128;           // 256 B rows of 16 hi | 16 lo tf32: 32 KB
constexpr int kRawW = BK * BN * 4;              // raw W rows: 32 x 256 fp32 = 32 KB
static_assert(BM == kRowsPerCta, "one TMEM lane per row");
constexpr int kRawBytes = kRawW + kRawDy;
constexpr int kOffRaw = kStages * kStageBytes;  // 96 KB
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
constexpr int kBN = BKH / (kXfThreads / BN);     // B elements per thread and half chunk: 8
constexpr int kACols = BKH / (kXfWarps / 4);     // A columns per transform warp: 4
static_assert(kBN == 8 && kACols == 4, "transform split");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol0 = 256;  // A operand slots: stage s hi at 256 + 32s, lo at +16
static_assert(kACol0 + 32 * kStages <= kTmemCols, "TMEM budget");

__host__ __device__ constexpr size_t dgrad_smem_bytes(int E) {
  return static_cast<size_t>(kOffTable) + sizeof(int) * (3 * static_cast<size_t>(E) + 3) + 1024;
}
static_assert(dgrad_smem_bytes(kMaxExperts) <= 232448, "shared memory budget");

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::tf32 (A: M rows in TMEM lanes, K in columns).
__device__ __forceinline__ void mma_tf32_at(uint32_t d, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) grouped_dgrad_kernel(const __grid_constant__ DgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int E = args.E, out_f = args.out_f, in_f = args.in_f;
  int* s_misc = reinterpret_cast<int*>(smem + kOffMisc);  // [0] tmem [1] abort [2] flag
  int* s_off = reinterpret_cast<int*>(smem + kOffTable);
  int* s_pad = s_off + (E + 1);
  int* s_rtp = s_pad + (E + 1);  // prefix of row-tile counts, E+1 entries
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&s_misc[1]);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane = lane_id();

  const uint32_t bar0 = sbase + kOffBar;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto bar_raw_full = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
  auto bar_raw_empty = [&](int s) { return bar0 + 8u * (2 * kStages + kRawStages + s); };
  const uint32_t bar_acc_full = bar0 + 8u * (2 * kStages + 2 * kRawStages);
  const uint32_t bar_acc_empty = bar_acc_full + 8u;
  const uint32_t bar_done = bar_acc_full + 16u;
  // Barriers, TMEM and the tensor maps are set up while the offsets are read (after an L2
  // flush that read is a DRAM round trip).
  if (tid == 0) {
    s_misc[1] = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full(s), kXfWarps);
      mbar_init(bar_empty(s), 1);
    }
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(bar_raw_full(s), 1);
      mbar_init(bar_raw_empty(s), kXfWarps);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, kEpiWarps);
    mbar_init(bar_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&args.tm_w);
    tma_prefetch_desc(&args.tm_dy);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_misc[0]), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  const bool offsets_ok = load_offsets(args.expert_off, E, args.rows, s_off, s_pad, &s_misc[2], args.status);
  tc_fence_after();  // load_offsets ends with a block barrier
  const uint32_t tmem = static_cast<uint32_t>(s_misc[0]);
  if (!offsets_ok) {
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  // Row tiles per expert = P-scan / 128 (the padded starts count ceil128 rows).
  for (int e = tid; e <= E; e += kThreads) s_rtp[e] = s_pad[e] / BM;
  __syncthreads();

  const int tiles_k = in_f / BN;
  const long long total = static_cast<long long>(s_rtp[E]) * tiles_k;
  const int nchunks = out_f / BK;

  if (warp == kTmaWarp) {
    // ---------------------------------------------- raw W and dy tiles by TMA
    if (lane == 0) {
      int rs = 0;
      uint32_t rph = 0;
      int pending[kRawStages];
      uint32_t pending_phase[kRawStages];
      for (int s = 0; s < kRawStages; ++s) pending[s] = 0, pending_phase[s] = 0;
      bool ok = true;
      bool dropped = false;
      // L2 prefetch cursor over this CTA's (item, chunk) sequence, kPrefetch chunks ahead of
      // the loads: the two-stage ring alone leaves each load a DRAM round trip to hide.
      long long pf_it = blockIdx.x;
      int pf_c = 0, pf_row0 = 0;
      Item pf_item{0, 0, 0};
      auto pf_set = [&]() {
        if (pf_it < total) {
          pf_item = decode_item(pf_it, tiles_k, s_rtp, E);
          pf_row0 = s_off[pf_item.e] + pf_item.rt * BM;
        }
      };
      auto pf_advance = [&](bool prefetch) {
        if (pf_it >= total) return;
        if (prefetch) {
          tma_prefetch_l2_2d(&args.tm_w, pf_item.kt * BN, pf_item.e * out_f + pf_c * BK);
          tma_prefetch_l2_2d(&args.tm_dy, pf_c * BK, pf_row0);
        }
        if (++pf_c == nchunks) {
          pf_c = 0;
          pf_it += gridDim.x;
          pf_set();
        }
      };
      pf_set();
      // The ring's first loads go out before any prefetch (the TMA unit serves them in
      // order); the cursor then starts past them and catches up two chunks per load.
      for (int i = 0; i < kRawStages; ++i) pf_advance(false);
      int ahead = kRawStages;
      for (long long it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const Item item = decode_item(it, tiles_k, s_rtp, E);
        const int row0 = s_off[item.e] + item.rt * BM;
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
                                   (item.kt + 1) * BN <= in_f && (c + 1) * BK <= out_f &&
                                   row0 < args.rows,
                               args.status);
          tma_load_2d(dst, &args.tm_w, item.kt * BN, item.e * out_f + c * BK, fb);
          tma_load_2d(dst + kRawW, &args.tm_dy, c * BK, row0, fb);
          --ahead;
          for (int k = 0; k < 2 && ahead < kPrefetch; ++k, ++ahead) pf_advance(true);
          pending[rs] = 1;
          pending_phase[rs] = rph;
          if (++rs == kRawStages) rs = 0, rph ^= 1u;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        if (args.status) atomicOr(args.status, kDevTimeout);
      }
      for (int s = 0; s < kRawStages; ++s)
        if (pending[s]) mbar_wait_drain(bar_raw_full(s), pending_phase[s]);
    }
  } else if (warp >= kXfWarp0) {
    // ----------------------------------------------------------- transform
    const int xw = warp - kXfWarp0;              // 0..15
    const int xt = tid - kXfWarp0 * 32;          // 0..511
    const int bk = xt % BN;                      // the B row k of this thread
    const int part = xt / BN;                    // its 8 of the half chunk's 16 n
    const uint32_t q = static_cast<uint32_t>(warp & 3);  // TMEM lane quarter for A
    const int kh = xw >> 2;                      // A columns 4*kh .. 4*kh+3 of a half chunk
    const uint32_t sw_b = static_cast<uint32_t>(bk & 7);  // 128B swizzle of B row bk
    int stage = 0, rs = 0;
    uint32_t phase = 0, rph = 0;
    bool ok = true;
    for (long long it = blockIdx.x; it < total && ok; it += gridDim.x) {
      for (int c = 0; c < nchunks; ++c) {
        if (!mbar_wait(bar_raw_full(rs), rph, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t raw_w = sbase + kOffRaw + rs * kRawBytes;
        const uint32_t raw_dy = raw_w + kRawW;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // W[n][k] for n = 16h + 8part + j of the chunk: column bk of the raw [32 n][256 k]
          // tile (a warp reads 32 consecutive k: conflict-free)
          float w[kBN];
#pragma unroll
          for (int j = 0; j < kBN; ++j)
            w[j] = ld_shared_f32(raw_w + static_cast<uint32_t>(((BKH * h + kBN * part + j) * BN + bk) * 4));
          const float4 a = load_a(raw_dy, h, q, lane, kh);
          if (!mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // B row bk: hi in 16-byte chunks 0-3, lo in 4-7 (logical), 128B-swizzled
          {
            uint32_t hi[kBN], lo[kBN];
#pragma unroll
            for (int j = 0; j < kBN; ++j) tf32_split(w[j], hi[j], lo[j]);
            const uint32_t row = sbase + stage * kStageBytes + bk * 128;
            const uint32_t c0 = 2u * part;
            st_shared_u4(row + ((c0 ^ sw_b) << 4), hi[0], hi[1], hi[2], hi[3]);
            st_shared_u4(row + (((c0 + 1u) ^ sw_b) << 4), hi[4], hi[5], hi[6], hi[7]);
            st_shared_u4(row + (((c0 + 4u) ^ sw_b) << 4), lo[0], lo[1], lo[2], lo[3]);
            st_shared_u4(row + (((c0 + 5u) ^ sw_b) << 4), lo[4], lo[5], lo[6], lo[7]);
          }
          // A hi/lo into this stage's TMEM slot, this warp's lane quarter and 4-column group
          store_a(a, q, kh, tmem, kACol0 + 32u * stage);
          tmem_wait_st();
          fence_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_full(stage));
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        // both halves of the raw stage are read
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_raw_empty(rs));
        if (++rs == kRawStages) rs = 0, rph ^= 1u;
      }
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0 && args.status) atomicOr(args.status, kDevTimeout);
    }
  } else {
    // ---------------------------------------- MMA issuer (warp 0, lane 0) and epilogue
    const int quarter = warp;  // warps 0-3
    const bool issuer = warp == 0 && lane == 0;
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    constexpr uint32_t idesc = idesc_tf32(BM, BN);
    const uint64_t b_desc0 = sdesc_kmajor_sw128(sbase);
    const int nhalves = 2 * nchunks;
    for (long long it = blockIdx.x; it < total; it += gridDim.x) {
      if (issuer && ok) {
        // the previous item's epilogue (all four warps) has read the accumulator
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
            mma_tf32_at(tmem, alo + 8u * ks, bhi + 2 * ks, idesc, (hc | ks) != 0);
            mma_tf32_at(tmem, ahi + 8u * ks, blo + 2 * ks, idesc, 1u);
            mma_tf32_at(tmem, ahi + 8u * ks, bhi + 2 * ks, idesc, 1u);
          }
          mma_commit(bar_empty(stage));
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
        if (ok) {
          mma_commit(bar_acc_full);
        } else {
          *abort_flag = 1;
          if (args.status) atomicOr(args.status, kDevTimeout);
        }
      }
      __syncwarp();
      if (*abort_flag) break;
      const uint64_t t_wait = MGW_DIAG_NOW();
      if (!mbar_wait(bar_acc_full, acc_phase, abort_flag)) {
        *abort_flag = 1;
        if (lane == 0 && args.status) atomicOr(args.status, kDevTimeout);
        break;
      }
      acc_phase ^= 1u;
      tc_fence_after();
      const Item item = decode_item(it, tiles_k, s_rtp, E);
      const int row0 = s_off[item.e] + item.rt * BM;
      const int valid = min(BM, s_off[item.e + 1] - row0);
      store_acc_rows(args, tmem, quarter, lane, row0, valid, item.kt * BN, BN);
      if (warp == 0 && lane == 0) MGW_DIAG_ITEM(dgrad, it, t_wait, MGW_DIAG_NOW());
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acc_empty);
    }
    if (issuer) {
      mma_commit(bar_done);
      mbar_wait_drain(bar_done, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_grouped_dgrad(const DgradArgs& a, int num_sms, cudaStream_t stream) {
  static thread_local uint64_t attr_ctx = 0;
  cudaError_t err = set_smem_attr_once(reinterpret_cast<const void*>(grouped_dgrad_kernel),
                                       dgrad_smem_bytes(kMaxExperts), &attr_ctx);
  if (err != cudaSuccess) return err;
  // Upper bound of the item count without reading expert_off on the host:
  // sum_e ceil(cnt_e/128) <= rows/128 + E.
  const long long max_items = (static_cast<long long>(a.rows) / BM + a.E) * (a.in_f / BN);
  long long grid = num_sms;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  grouped_dgrad_kernel<<<static_cast<unsigned>(grid), kThreads, dgrad_smem_bytes(a.E), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mgw
