// Grouped fp32 data gradient with 3xTF32 tcgen05 MMAs.
//
//   dx[r, k] = sum_n dy[r, n] * W[e(r), n, k],  e(r): the expert whose row range holds r.
//
// Work item = (expert e, 128-row tile inside e's row range, 256-column k tile).
// Tiles start at expert_off[e], so a tile never mixes experts: rows of the tile
// past the expert's last row are loaded as zero and never stored.  This replaces
// the dgrad page's split between a tiled path and a per-element path for tiles
// that straddle an expert boundary.
//
// Precision: each fp32 operand x is split as hi = tf32(x), lo = tf32(x - hi)
// (both rounded with cvt.rna.tf32), and the product is hi*hi + hi*lo + lo*hi
// accumulated in fp32 in TMEM (Ootomo & Yokota, "Recovering single precision
// accuracy from Tensor Cores while surpassing the FP32 theoretical peak
// performance", IJHPCA 2022).
//
// Data path per 32-wide reduction chunk:
//   * W[e] rows n (32 of them, 256 k columns) arrive raw by TMA into a two-stage ring;
//   * the transform warps split them into hi/lo and write the MMA's B operand transposed
//     (K-major, 128B-swizzled) into a two-stage shared-memory ring, and split the chunk's
//     dy rows (loaded straight into registers) into hi/lo A operands that they store into
//     TMEM with tcgen05.st, so A never occupies shared memory;
//   * the MMA thread issues 4 K-steps x 3 tcgen05.mma.kind::tf32 (M=128, N=256, K=8)
//     with A from TMEM and B from shared memory into one 256-column accumulator.
//
// Roles (704 threads):
//   warps 0-3   epilogue: TMEM lane quarter = warp, 32-column chunks -> fp32 stores of
//               the rows that belong to the item's expert, then the accumulator is free.
//   warp 4      MMA issuer.
//   warps 5-20  transform: per chunk, thread t splits half of B row t % 256 (16 of the 32
//               reduction elements) and 8 A elements of one row (four warps per TMEM lane
//               quarter, 8 columns each).  Sixteen warps instead of eight halve each warp's
//               serial chain of loads, splits and stores per chunk.
//   warp 21     TMA producer of the raw W tiles.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace mgw {
namespace {

constexpr int BM = 128;  // rows per tile (MMA M)
constexpr int BN = 256;  // dx columns per tile (MMA N)
constexpr int BK = 32;   // reduction (out_features) per stage: one 128-byte row of fp32
constexpr int kStages = 2;
constexpr int kRawStages = 2;
constexpr int kBTile = BN * BK * 4;             // 32 KB (hi or lo)
constexpr int kStageBytes = 2 * kBTile;         // B_hi, B_lo = 64 KB
constexpr int kRawBytes = BK * BN * 4;          // raw W rows: 32 x 256 fp32 = 32 KB
constexpr int kOffRaw = kStages * kStageBytes;  // 128 KB
constexpr int kOffBar = kOffRaw + kRawStages * kRawBytes;
// full[], empty[], raw_full[], raw_empty[], acc_full, acc_empty, done
constexpr int kNumBars = 2 * kStages + 2 * kRawStages + 3;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffTable = kOffMisc + 16;
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kXfWarp0 = 5;
constexpr int kXfWarps = 16;
constexpr int kXfThreads = kXfWarps * 32;
constexpr int kBParts = kXfThreads / BN;     // threads per B row
constexpr int kNgPer = (BK / 4) / kBParts;   // groups of 4 reduction elements per thread
constexpr int kACols = BK / (kXfWarps / 4);  // A columns per transform warp
constexpr int kTmaWarp = kXfWarp0 + kXfWarps;
constexpr int kThreads = (kTmaWarp + 1) * 32;
static_assert(kXfThreads % BN == 0 && (BK / 4) % kBParts == 0 && kACols == 8, "transform split");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol0 = 256;  // A operand slots: stage s hi at 256 + 64s, lo at +32

__host__ __device__ constexpr size_t dgrad_smem_bytes(int E) {
  return static_cast<size_t>(kOffTable) + sizeof(int) * (3 * static_cast<size_t>(E) + 3) + 1024;
}
static_assert(dgrad_smem_bytes(kMaxExperts) <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void split1(float v, uint32_t& hi, uint32_t& lo) {
  hi = tf32_rna(v);
  lo = tf32_rna(v - __uint_as_float(hi));
}

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

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::tf32 (A: M rows in TMEM lanes, K in columns).
__device__ __forceinline__ void mma_tf32_at(uint32_t d, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  int never = 0;
  (void)mbar_wait(bar, parity, &never);
}

// Item it -> (expert, row tile in expert, k tile) via the prefix of row-tile counts.
struct Item {
  int e, rt, kt;
};
__device__ __forceinline__ Item decode_item(long long it, int tiles_k, const int* s_rtp, int E) {
  const int t = static_cast<int>(it / tiles_k);
  Item r;
  r.kt = static_cast<int>(it % tiles_k);
  int lo = 0, hi = E - 1;  // largest e with s_rtp[e] <= t (a non-empty expert)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_rtp[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  r.e = lo;
  r.rt = t - s_rtp[lo];
  return r;
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

  if (tid == 0) s_misc[1] = 0;
  if (!load_offsets(args.expert_off, E, args.rows, s_off, s_pad, &s_misc[2], args.status)) return;
  // Row tiles per expert = P-scan / 128 (the padded starts count ceil128 rows).
  for (int e = tid; e <= E; e += kThreads) s_rtp[e] = s_pad[e] / BM;

  const uint32_t bar0 = sbase + kOffBar;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto bar_raw_full = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
  auto bar_raw_empty = [&](int s) { return bar0 + 8u * (2 * kStages + kRawStages + s); };
  const uint32_t bar_acc_full = bar0 + 8u * (2 * kStages + 2 * kRawStages);
  const uint32_t bar_acc_empty = bar_acc_full + 8u;
  const uint32_t bar_done = bar_acc_full + 16u;
  if (tid == 0) {
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
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&s_misc[0]), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(s_misc[0]);

  const int tiles_k = in_f / BN;
  const long long total = static_cast<long long>(s_rtp[E]) * tiles_k;
  const int nchunks = out_f / BK;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------- raw W tiles by TMA
    if (lane == 0) {
      int rs = 0;
      uint32_t rph = 0;
      int pending[kRawStages];
      uint32_t pending_phase[kRawStages];
      for (int s = 0; s < kRawStages; ++s) pending[s] = 0, pending_phase[s] = 0;
      bool ok = true;
      for (long long it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const Item item = decode_item(it, tiles_k, s_rtp, E);
        for (int c = 0; c < nchunks; ++c) {
          if (!mbar_wait(bar_raw_empty(rs), rph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_raw_full(rs);
          mbar_arrive_expect_tx(fb, kRawBytes);
          tma_load_2d(sbase + kOffRaw + rs * kRawBytes, &args.tm_w, item.kt * BN,
                      item.e * out_f + c * BK, fb);
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
    const int ng0 = (xt / BN) * kNgPer;          // its first group of 4 reduction elements
    const uint32_t q = static_cast<uint32_t>(warp & 3);  // TMEM lane quarter for A
    const int kh = xw >> 2;                      // A columns 8*kh .. 8*kh+7 of the chunk
    int stage = 0, rs = 0;
    uint32_t phase = 0, rph = 0;
    bool ok = true;
    for (long long it = blockIdx.x; it < total && ok; it += gridDim.x) {
      const Item item = decode_item(it, tiles_k, s_rtp, E);
      const int row0 = s_off[item.e] + item.rt * BM;
      const int valid = min(BM, s_off[item.e + 1] - row0);
      const int r = static_cast<int>(q) * 32 + static_cast<int>(lane);  // this thread's A row
      const float* dyrow = args.dy + static_cast<size_t>(row0 + (r < valid ? r : 0)) * out_f + kACols * kh;
      for (int c = 0; c < nchunks; ++c) {
        // A: 8 consecutive reduction elements of row r, straight from global memory
        float4 a4[kACols / 4];
#pragma unroll
        for (int j = 0; j < kACols / 4; ++j) {
          a4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (r < valid) a4[j] = __ldg(reinterpret_cast<const float4*>(dyrow + c * BK) + j);
        }
        if (!mbar_wait(bar_raw_full(rs), rph, abort_flag) ||
            !mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        // B: row k = bk of the K-major tile holds W[n][k] for the chunk's 32 n; this thread
        // reads its half of column k of the raw [32 n][256 k] tile (conflict-free) and writes
        // 4 x 16 bytes of each of the hi and lo rows
        const float* raw = reinterpret_cast<const float*>(smem + kOffRaw + rs * kRawBytes);
        const uint32_t s_bhi = sbase + stage * kStageBytes;
        const uint32_t s_blo = s_bhi + kBTile;
#pragma unroll
        for (int g = 0; g < kNgPer; ++g) {
          const int ng = ng0 + g;
          uint32_t h[4], l[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) split1(raw[(4 * ng + j) * BN + bk], h[j], l[j]);
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
            split1(a4[j].x, ah[4 * j], al[4 * j]);
            split1(a4[j].y, ah[4 * j + 1], al[4 * j + 1]);
            split1(a4[j].z, ah[4 * j + 2], al[4 * j + 2]);
            split1(a4[j].w, ah[4 * j + 3], al[4 * j + 3]);
          }
          const uint32_t ta = tmem + (q * 32u << 16) + kACol0 + 64u * stage + kACols * kh;
          tmem_st_x8(ta, ah);
          tmem_st_x8(ta + 32, al);
          tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_full(stage));
        if (++stage == kStages) stage = 0, phase ^= 1u;
      }
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0 && args.status) atomicOr(args.status, kDevTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      constexpr uint32_t idesc = idesc_tf32(BM, BN);
      const uint64_t b_desc0 = sdesc_kmajor_sw128(sbase);
      for (long long it = blockIdx.x; it < total && ok; it += gridDim.x) {
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
          const uint64_t bhi = b_desc0 + static_cast<uint32_t>(stage * (kStageBytes >> 4));
          const uint64_t blo = bhi + (kBTile >> 4);
          const uint32_t ahi = tmem + kACol0 + 64u * stage;
          const uint32_t alo = ahi + 32u;
#pragma unroll
          for (int ks = 0; ks < BK / 8; ++ks) {
            mma_tf32_at(tmem, alo + 8u * ks, bhi + 2 * ks, idesc, (c | ks) != 0);
            mma_tf32_at(tmem, ahi + 8u * ks, blo + 2 * ks, idesc, 1u);
            mma_tf32_at(tmem, ahi + 8u * ks, bhi + 2 * ks, idesc, 1u);
          }
          mma_commit(bar_empty(stage));
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit(bar_acc_full);
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
    const int quarter = warp;  // warps 0-3
    uint32_t acc_phase = 0;
    for (long long it = blockIdx.x; it < total; it += gridDim.x) {
      if (*abort_flag) break;
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
      const int r = quarter * 32 + static_cast<int>(lane);
      float* dst = args.dx + static_cast<size_t>(row0 + r) * in_f + item.kt * BN;
      const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int j = 0; j < BN / 32; ++j) {
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
      if (lane == 0) mbar_arrive(bar_acc_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
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
