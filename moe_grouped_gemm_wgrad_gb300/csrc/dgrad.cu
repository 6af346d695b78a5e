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
// Roles (416 threads):
//   warps 0-3   epilogue: TMEM lane quarter = warp, 32-column chunks -> fp32
//               stores of the rows that belong to the item's expert.
//   warp 4      MMA issuer: per 32-wide reduction chunk, 4 K-steps x 3
//               tcgen05.mma.kind::tf32 (M=128, N=256, K=8) into one of two TMEM
//               accumulators (2 x 256 columns), so the epilogue of one item
//               overlaps the main loop of the next.
//   warps 5-12  transform: load dy and W tiles from global memory one chunk ahead
//               (software pipelined in registers; the chunk after that is prefetched
//               into L2), split into hi/lo, write K-major
//               128B-swizzled tiles (W transposed on the fly) into a 2-stage
//               shared-memory ring.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace mgw {
namespace {

constexpr int BM = 128;  // rows per tile (MMA M)
constexpr int BN = 256;  // dx columns per tile (MMA N)
constexpr int BK = 32;   // reduction (out_features) per stage: one 128-byte row of fp32
constexpr int kStages = 2;
constexpr int kATile = BM * BK * 4;                 // 16 KB
constexpr int kBTile = BN * BK * 4;                 // 32 KB
constexpr int kStageBytes = 2 * kATile + 2 * kBTile;  // A_hi, A_lo, B_hi, B_lo = 96 KB
constexpr int kOffBar = kStages * kStageBytes;
constexpr int kNumBars = 2 * kStages + 4 + 1;  // full[], empty[], acc_full[2], acc_empty[2], done
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffTable = kOffMisc + 16;
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kXfWarps = 8;
constexpr int kThreads = (kEpiWarps + 1 + kXfWarps) * 32;
constexpr uint32_t kTmemCols = 512;
// Chunks between the one loaded into registers and the one prefetched into L2.
constexpr int kPrefetchAhead = 1;

__host__ __device__ constexpr size_t dgrad_smem_bytes(int E) {
  return static_cast<size_t>(kOffTable) + sizeof(int) * (3 * static_cast<size_t>(E) + 3) + 1024;
}
static_assert(dgrad_smem_bytes(kMaxExperts) <= 232448, "shared memory budget");

__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void split4(const float4& v, uint4& hi, uint4& lo) {
  hi.x = tf32_rna(v.x);
  hi.y = tf32_rna(v.y);
  hi.z = tf32_rna(v.z);
  hi.w = tf32_rna(v.w);
  lo.x = tf32_rna(v.x - __uint_as_float(hi.x));
  lo.y = tf32_rna(v.y - __uint_as_float(hi.y));
  lo.z = tf32_rna(v.z - __uint_as_float(hi.z));
  lo.w = tf32_rna(v.w - __uint_as_float(hi.w));
}

__device__ __forceinline__ void st_shared_u4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
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
  auto bar_acc_full = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto bar_acc_empty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t bar_done = bar0 + 8u * (2 * kStages + 4);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full(s), kXfWarps);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full(b), 1);
      mbar_init(bar_acc_empty(b), kEpiWarps);
    }
    mbar_init(bar_done, 1);
    fence_mbar_init();
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

  if (warp >= kEpiWarps + 1) {
    // ----------------------------------------------------------- transform
    // Software-pipelined: the global loads of the next chunk (possibly of the next item)
    // are in flight while the current chunk is split and written to shared memory.
    const int xt = tid - (kEpiWarps + 1) * 32;  // 0..255
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // raw operands of one chunk in registers: dy 4 x float4, W 8 x 4 floats
    struct Raw {
      float4 a[4];
      float b[8][4];
    };
    auto load_chunk = [&](const Item& item, int c, Raw& raw) {
      const int row0 = s_off[item.e] + item.rt * BM;
      const int valid = min(BM, s_off[item.e + 1] - row0);
      // A = dy[row0 .. row0+127, 32c .. 32c+31]: 128 rows x 8 chunks of 16 B.
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int idx = xt + p * 256;
        const int r = idx >> 3, j = idx & 7;
        raw.a[p] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < valid)
          raw.a[p] = __ldg(reinterpret_cast<const float4*>(
              args.dy + static_cast<size_t>(row0 + r) * out_f + c * BK + 4 * j));
      }
      // B^T tile: dx column k (K-major row k of B) and 4 consecutive n; lane -> k.
      const float* Wk = args.W + static_cast<size_t>(item.e) * out_f * in_f + item.kt * BN;
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const int idx = xt + p * 256;            // 0..2047
        const int k = idx & 255, ng = idx >> 8;  // ng in 0..7
        const float* src = Wk + static_cast<size_t>(c * BK + 4 * ng) * in_f + k;
#pragma unroll
        for (int q = 0; q < 4; ++q) raw.b[p][q] = __ldg(src + static_cast<size_t>(q) * in_f);
      }
    };
    // L2 prefetch of a chunk: its 32 W row segments (8 lines each) and 128 dy row segments
    // (one line each), 384 lines over 256 threads, so that the register loads one chunk
    // later hit L2 instead of waiting on DRAM.
    auto prefetch_chunk = [&](const Item& item, int c) {
      const int row0 = s_off[item.e] + item.rt * BM;
      const int valid = min(BM, s_off[item.e + 1] - row0);
      const float* Wk = args.W + static_cast<size_t>(item.e) * out_f * in_f + item.kt * BN;
      for (int i = xt; i < 384; i += 256) {
        const float* p;
        if (i < 256) {
          p = Wk + static_cast<size_t>(c * BK + (i >> 3)) * in_f + (i & 7) * 32;
        } else {
          const int r = i - 256;
          if (r >= valid) continue;
          p = args.dy + static_cast<size_t>(row0 + r) * out_f + c * BK;
        }
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
      }
    };
    // (item, c) -> the chunk after it in this CTA's sequence; false past the last
    auto advance = [&](long long& it2, Item& item2, int& c2) -> bool {
      if (++c2 == nchunks) {
        c2 = 0;
        it2 += gridDim.x;
        if (it2 >= total) return false;
        item2 = decode_item(it2, tiles_k, s_rtp, E);
      }
      return true;
    };
    long long it = blockIdx.x;
    Raw cur, nxt;
    Item item{0, 0, 0};
    int c = 0;
    if (it < total) {
      item = decode_item(it, tiles_k, s_rtp, E);
      load_chunk(item, 0, cur);
    }
    while (it < total && ok) {
      // the chunk after (item, c): next chunk of this item, else chunk 0 of the next item
      long long nit = it;
      int nc = c + 1;
      Item nitem = item;
      if (nc == nchunks) {
        nc = 0;
        nit = it + gridDim.x;
        if (nit < total) nitem = decode_item(nit, tiles_k, s_rtp, E);
      }
      if (nit < total) {
        load_chunk(nitem, nc, nxt);
        long long pit = nit;
        Item pitem = nitem;
        int pc = nc;
        bool more = true;
        for (int d = 0; d < kPrefetchAhead && more; ++d) more = advance(pit, pitem, pc);
        if (more) prefetch_chunk(pitem, pc);
      }
      if (!mbar_wait(bar_empty(stage), phase ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      const uint32_t s_ahi = sbase + stage * kStageBytes;
      const uint32_t s_alo = s_ahi + kATile;
      const uint32_t s_bhi = s_alo + kATile;
      const uint32_t s_blo = s_bhi + kBTile;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int idx = xt + p * 256;
        const int r = idx >> 3, j = idx & 7;
        uint4 hi, lo;
        split4(cur.a[p], hi, lo);
        const uint32_t off = r * 128 + ((j ^ (r & 7)) << 4);
        st_shared_u4(s_ahi + off, hi);
        st_shared_u4(s_alo + off, lo);
      }
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const int idx = xt + p * 256;
        const int k = idx & 255, ng = idx >> 8;
        uint4 hi, lo;
        split4(make_float4(cur.b[p][0], cur.b[p][1], cur.b[p][2], cur.b[p][3]), hi, lo);
        const uint32_t off = k * 128 + ((ng ^ (k & 7)) << 4);
        st_shared_u4(s_bhi + off, hi);
        st_shared_u4(s_blo + off, lo);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_full(stage));
      if (++stage == kStages) stage = 0, phase ^= 1u;
      it = nit;
      c = nc;
      item = nitem;
      cur = nxt;
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0 && args.status) atomicOr(args.status, kDevTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase[2] = {0u, 0u};
      int local = 0;
      bool ok = true;
      constexpr uint32_t idesc = idesc_tf32(BM, BN);
      const uint64_t a_desc0 = sdesc_kmajor_sw128(sbase);
      for (long long it = blockIdx.x; it < total && ok; it += gridDim.x, ++local) {
        const int b = local & 1;
        if (!mbar_wait_spin(bar_acc_empty(b), acc_phase[b] ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        acc_phase[b] ^= 1u;
        tc_fence_after();
        const uint32_t dacc = tmem + 256u * b;
        for (int c = 0; c < nchunks; ++c) {
          if (!mbar_wait_spin(bar_full(stage), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors from one base: tiles and the 32-byte K steps are offsets / 16 in the
          // start-address field (the ring lies below 256 KB: no carry)
          const uint64_t ahi = a_desc0 + static_cast<uint32_t>(stage * (kStageBytes >> 4));
          const uint64_t alo = ahi + (kATile >> 4);
          const uint64_t bhi = alo + (kATile >> 4);
          const uint64_t blo = bhi + (kBTile >> 4);
#pragma unroll
          for (int ks = 0; ks < BK / 8; ++ks) {
            mma_tf32(dacc, alo + 2 * ks, bhi + 2 * ks, idesc, (c | ks) != 0);
            mma_tf32(dacc, ahi + 2 * ks, blo + 2 * ks, idesc, 1u);
            mma_tf32(dacc, ahi + 2 * ks, bhi + 2 * ks, idesc, 1u);
          }
          mma_commit(bar_empty(stage));
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit(bar_acc_full(b));
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
    uint32_t acc_phase[2] = {0u, 0u};
    int local = 0;
    for (long long it = blockIdx.x; it < total; it += gridDim.x, ++local) {
      const int b = local & 1;
      if (*abort_flag) break;
      if (!mbar_wait(bar_acc_full(b), acc_phase[b], abort_flag)) {
        *abort_flag = 1;
        if (lane == 0 && args.status) atomicOr(args.status, kDevTimeout);
        break;
      }
      acc_phase[b] ^= 1u;
      tc_fence_after();
      const Item item = decode_item(it, tiles_k, s_rtp, E);
      const int row0 = s_off[item.e] + item.rt * BM;
      const int valid = min(BM, s_off[item.e + 1] - row0);
      const int r = quarter * 32 + static_cast<int>(lane);
      float* dst = args.dx + static_cast<size_t>(row0 + r) * in_f + item.kt * BN;
      const uint32_t ta = tmem + 256u * b + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int j = 0; j < BN / 32; ++j) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(ta + 32u * j, v);
        tmem_wait_ld();
        if (r < valid) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(dst + 32 * j + 4 * q) =
                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acc_empty(b));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_grouped_dgrad(const DgradArgs& a, int num_sms, cudaStream_t stream) {
  static thread_local int attr_set_device = -1;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (attr_set_device != dev) {
    err = cudaFuncSetAttribute(grouped_dgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(dgrad_smem_bytes(kMaxExperts)));
    if (err != cudaSuccess) return err;
    attr_set_device = dev;
  }
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
