// C ABI of libmgw.so (declared in include/mgw.h): argument checks, TMA tensor
// maps, device checks and kernel launches.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/mgw.h"
#ifdef MGW_DIAG
#include "../../include/mgw_diag.h"
#endif
#include "kernels.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

// Checks that the current device is compute capability 10.3 and returns its SM count.
mgw_status current_device(DeviceInfo* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MGW_ERR_CUDA;
  static DeviceInfo cache[64];
  static std::mutex mu;
  if (dev < 0 || dev >= 64) return MGW_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev].ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MGW_ERR_CUDA;
    if (major != 10 || minor != 3) return MGW_ERR_ARCH;
    cache[dev].sms = sms;
    cache[dev].ok = true;
  }
  *info = cache[dev];
  return MGW_OK;
}

// A tensor map is plain data (base address, sizes, strides, box and swizzle), so encoded
// maps are kept in a small process-wide table keyed by every one of those inputs and reused
// by later calls on the same buffers.
struct MapKey {
  const void* base;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  int rank, dt, swz;
  bool operator==(const MapKey& o) const {
    return base == o.base && rank == o.rank && dt == o.dt && swz == o.swz &&
           std::memcmp(dims, o.dims, sizeof(dims)) == 0 &&
           std::memcmp(strides, o.strides, sizeof(strides)) == 0 &&
           std::memcmp(box, o.box, sizeof(box)) == 0;
  }
};
constexpr int kMapCacheSize = 64;
struct MapCache {
  std::mutex mu;
  MapKey key[kMapCacheSize];
  CUtensorMap map[kMapCacheSize];
  int used = 0, next = 0;
};
MapCache& map_cache() {
  static MapCache c;
  return c;
}

// Tiled tensor map of rank 2 or 3: dims[0] contiguous elements, strides in bytes of dims 1, 2.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank,
              const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
              CUtensorMapSwizzle swz) {
  MapKey k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.rank = rank;
  k.dt = static_cast<int>(dt);
  k.swz = static_cast<int>(swz);
  for (int i = 0; i < rank; ++i) k.dims[i] = dims[i], k.box[i] = box[i];
  for (int i = 0; i + 1 < rank; ++i) k.strides[i] = strides[i];
  MapCache& c = map_cache();
  {
    std::lock_guard<std::mutex> lock(c.mu);
    for (int i = 0; i < c.used; ++i)
      if (c.key[i] == k) {
        *m = c.map[i];
        return true;
      }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], estr[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) gd[i] = dims[i], bx[i] = box[i];
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides[i];
  std::memset(m, 0, sizeof(*m));
  if (fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(c.mu);
  const int slot = c.used < kMapCacheSize ? c.used++ : (c.next++ % kMapCacheSize);
  c.key[slot] = k;
  c.map[slot] = *m;
  return true;
}

// 2-D tiled tensor map: `inner` contiguous elements per row, `outer` rows, `pitch` bytes
// between rows.
bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t pitch, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swz) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {pitch};
  const uint32_t box[2] = {box_inner, box_outer};
  return make_map(m, dt, base, 2, dims, strides, box, swz);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace mgw {

uint64_t current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return static_cast<uint64_t>(id);
}

cudaError_t set_smem_attr_once(const void* kernel, size_t bytes, uint64_t* done_ctx) {
  const uint64_t id = current_context_id();
  if (id != 0 && id == *done_ctx) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(bytes));
  if (err != cudaSuccess) return err;
  // The call above made the device's context current if no context was.
  *done_ctx = current_context_id();
  return cudaSuccess;
}

}  // namespace mgw

extern "C" {

const char* mgw_status_string(mgw_status s) {
  switch (s) {
    case MGW_OK: return "ok";
    case MGW_ERR_INVALID_ARG: return "invalid argument";
    case MGW_ERR_UNSUPPORTED: return "unsupported size";
    case MGW_ERR_CAPACITY: return "padded token capacity too small or not a multiple of 128";
    case MGW_ERR_CUDA: return "CUDA error";
    case MGW_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    default: return "unknown status";
  }
}

int mgw_version(void) { return 100; }

size_t mgw_mxfp8_token_capacity(int M, int E) {
  if (M < 0 || E < 1) return 0;
  const size_t need = static_cast<size_t>(M) + 127u * static_cast<size_t>(E);
  return (need + 127u) / 128u * 128u;
}

size_t mgw_mxfp8_scale_bytes(int C, size_t Mcap) {
  if (C < 0) return 0;
  return static_cast<size_t>(C) * Mcap / 32u;
}

}  // extern "C"

namespace {

mgw_status quantize_impl(const void* src_bf16, int src_rows, const int32_t* row_index, int M,
                         int C, const int32_t* expert_off, int E, void* q_e4m3,
                         void* scales_e8m0, size_t Mcap, int scale_rule, int* status_dev,
                         void* stream) {
  if (!expert_off || !q_e4m3 || !scales_e8m0 || (M > 0 && !src_bf16)) return MGW_ERR_INVALID_ARG;
  if (M < 0 || C <= 0 || E < 1 || E > MGW_MAX_EXPERTS) return MGW_ERR_INVALID_ARG;
  if (scale_rule != MGW_SCALE_FLOOR && scale_rule != MGW_SCALE_CEIL_448) return MGW_ERR_INVALID_ARG;
  if (row_index != nullptr && src_rows < 1) return MGW_ERR_INVALID_ARG;
  if (C % 128 != 0) return MGW_ERR_UNSUPPORTED;
  if (Mcap % 128 != 0 || Mcap < mgw_mxfp8_token_capacity(M, E) || Mcap > (size_t(1) << 31))
    return MGW_ERR_CAPACITY;
  if ((src_bf16 && !aligned16(src_bf16)) || !aligned16(q_e4m3) || !aligned16(scales_e8m0))
    return MGW_ERR_INVALID_ARG;
  DeviceInfo dev;
  mgw_status st = current_device(&dev);
  if (st != MGW_OK) return st;
  // Contiguous source: 128 x 128 tiles.  Gathered source: one-row boxes for tile::gather4.
  // With M == 0 the map is never used; it then only needs a valid address.
  CUtensorMap tm_src;
  const bool gather = M > 0 && row_index != nullptr;
  const bool tile_src = M > 0 && row_index == nullptr;
  const void* map_base = (gather || tile_src) ? src_bf16 : q_e4m3;
  const uint64_t map_rows = gather ? static_cast<uint64_t>(src_rows)
                                   : (tile_src ? static_cast<uint64_t>(M) : 1);
  if (!make_map_2d(&tm_src, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map_base, C, map_rows,
                   static_cast<uint64_t>(C) * 2, 128, gather ? 1 : 128, CU_TENSOR_MAP_SWIZZLE_NONE))
    return MGW_ERR_CUDA;
  CUtensorMap tm_q;
  if (!make_map_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_e4m3, Mcap, C, Mcap, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return MGW_ERR_CUDA;
  const cudaError_t err = mgw::launch_mxfp8_quantize(
      tm_src, tm_q, M, C, expert_off, E, scales_e8m0, static_cast<long long>(Mcap), scale_rule,
      status_dev, dev.sms, static_cast<cudaStream_t>(stream), src_bf16, row_index, src_rows);
  return err == cudaSuccess ? MGW_OK : MGW_ERR_CUDA;
}

}  // namespace

extern "C" {

mgw_status mgw_mxfp8_quantize(const void* src_bf16, int M, int C, const int32_t* expert_off,
                              int E, void* q_e4m3, void* scales_e8m0, size_t Mcap,
                              int scale_rule, int* status_dev, void* stream) {
  return quantize_impl(src_bf16, M, nullptr, M, C, expert_off, E, q_e4m3, scales_e8m0, Mcap,
                       scale_rule, status_dev, stream);
}

mgw_status mgw_mxfp8_quantize_gather(const void* src_bf16, int src_rows,
                                     const int32_t* row_index, int M, int C,
                                     const int32_t* expert_off, int E, void* q_e4m3,
                                     void* scales_e8m0, size_t Mcap, int scale_rule,
                                     int* status_dev, void* stream) {
  if (M > 0 && (!row_index || !src_bf16 || src_rows < 1)) return MGW_ERR_INVALID_ARG;
  return quantize_impl(src_bf16, src_rows, M > 0 ? row_index : nullptr, M, C, expert_off, E,
                       q_e4m3, scales_e8m0, Mcap, scale_rule, status_dev, stream);
}

}  // extern "C"

namespace {

mgw_status wgrad_check(const void* gq, const void* gs, const void* xq, const void* xs,
                       const int32_t* expert_off, int E, int M, int N, int K, size_t Mcap,
                       void* out_bf16) {
  if (!gq || !gs || !xq || !xs || !expert_off || !out_bf16) return MGW_ERR_INVALID_ARG;
  if (M < 0 || N <= 0 || K <= 0 || E < 1 || E > MGW_MAX_EXPERTS) return MGW_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 256 != 0) return MGW_ERR_UNSUPPORTED;
  if (static_cast<long long>(E) * N > (1ll << 31)) return MGW_ERR_UNSUPPORTED;
  // output tiles (128 x 256) must be countable in 32 bits
  if (static_cast<long long>(E) * (N / 128) * (K / 256) >= (1ll << 31)) return MGW_ERR_UNSUPPORTED;
  if (Mcap % 128 != 0 || Mcap < mgw_mxfp8_token_capacity(M, E) || Mcap > (size_t(1) << 31))
    return MGW_ERR_CAPACITY;
  if (!aligned16(gq) || !aligned16(xq) || !aligned16(gs) || !aligned16(xs) || !aligned16(out_bf16))
    return MGW_ERR_INVALID_ARG;
  return MGW_OK;
}

// Tensor maps and sizes of the wgrad kernels; `pair` selects the CTA-pair layout (x^T boxes
// of 128 rows, scale atoms loaded by TMA).
bool wgrad_maps(mgw::WgradArgs* a, const void* gq, const void* gs, const void* xq,
                const void* xs, const int32_t* expert_off, int E, int M, int N, int K,
                size_t Mcap, void* out_bf16, int* status_dev, bool pair) {
  std::memset(a, 0, sizeof(*a));
  if (!make_map_2d(&a->tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, gq, Mcap, N, Mcap, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&a->tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, Mcap, K, Mcap, 128,
                   pair ? 128 : 256, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&a->tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out_bf16, K,
                   static_cast<uint64_t>(E) * N, static_cast<uint64_t>(K) * 2, 64, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return false;
  // Scale atoms of the CTA-pair kernel as rows of 256 bytes (an atom is 2 rows).
  if (pair && (!make_map_2d(&a->tm_sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, gs, 256,
                            static_cast<uint64_t>(N) * (Mcap / 32) / 256, 256, 256, 2,
                            CU_TENSOR_MAP_SWIZZLE_NONE) ||
               !make_map_2d(&a->tm_sfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, xs, 256,
                            static_cast<uint64_t>(K) * (Mcap / 32) / 256, 256, 256, 4,
                            CU_TENSOR_MAP_SWIZZLE_NONE)))
    return false;
  a->out = out_bf16;
  a->gs = static_cast<const uint8_t*>(gs);
  a->xs = static_cast<const uint8_t*>(xs);
  a->expert_off = expert_off;
  a->E = E;
  a->M = M;
  a->N = N;
  a->K = K;
  a->mcap = static_cast<long long>(Mcap);
  a->status = status_dev;
  return true;
}

}  // namespace

extern "C" {

size_t mgw_grouped_wgrad_workspace_bytes(int E, int N, int K) {
  (void)E;
  (void)N;
  (void)K;
  DeviceInfo dev;
  if (current_device(&dev) != MGW_OK) return 0;
  return mgw::balanced_workspace_bytes(2 * dev.sms);
}

mgw_status mgw_grouped_wgrad_mxfp8_balanced(const void* gq, const void* gs, const void* xq,
                                            const void* xs, const int32_t* expert_off, int E,
                                            int M, int N, int K, size_t Mcap, void* out_bf16,
                                            void* workspace, size_t workspace_bytes,
                                            int* status_dev, void* stream) {
  mgw_status st = wgrad_check(gq, gs, xq, xs, expert_off, E, M, N, K, Mcap, out_bf16);
  if (st != MGW_OK) return st;
  if (E > mgw::kMaxBalancedExperts) return MGW_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MGW_ERR_INVALID_ARG;
  const int slots = mgw::balanced_workspace_slots(workspace_bytes);
  if (slots < 0) return MGW_ERR_CAPACITY;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != MGW_OK) return st;
  mgw::WgradArgs a;
  if (!wgrad_maps(&a, gq, gs, xq, xs, expert_off, E, M, N, K, Mcap, out_bf16, status_dev, false))
    return MGW_ERR_CUDA;
  const cudaError_t err = mgw::launch_grouped_wgrad_balanced(a, workspace, slots, dev.sms,
                                                             static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MGW_OK : MGW_ERR_CUDA;
}

mgw_status mgw_grouped_wgrad_mxfp8_balanced_noalloc(const void* gq, const void* gs,
                                                    const void* xq, const void* xs,
                                                    const int32_t* expert_off, int E, int M,
                                                    int N, int K, size_t Mcap, void* out_bf16,
                                                    int* status_dev, void* stream) {
  mgw_status st = wgrad_check(gq, gs, xq, xs, expert_off, E, M, N, K, Mcap, out_bf16);
  if (st != MGW_OK) return st;
  if (E > mgw::kMaxBalancedExperts) return MGW_ERR_UNSUPPORTED;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != MGW_OK) return st;
  void* ws = nullptr;
  size_t ws_bytes = 0, counter_bytes = 0;
  if (mgw::noalloc_wgrad_workspace(&ws, &ws_bytes, &counter_bytes) != cudaSuccess)
    return MGW_ERR_CUDA;
  const int slots = mgw::balanced_workspace_slots(ws_bytes);
  // The kernel leaves its counters at zero, but a call that ended with MGW_DEV_TIMEOUT may
  // not have: clear them (under 1 KB, on the call's stream) so every call starts clean.
  if (cudaMemsetAsync(ws, 0, counter_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MGW_ERR_CUDA;
  mgw::WgradArgs a;
  if (!wgrad_maps(&a, gq, gs, xq, xs, expert_off, E, M, N, K, Mcap, out_bf16, status_dev, false))
    return MGW_ERR_CUDA;
  const cudaError_t err = mgw::launch_grouped_wgrad_balanced(a, ws, slots, dev.sms,
                                                             static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MGW_OK : MGW_ERR_CUDA;
}

mgw_status mgw_grouped_wgrad_mxfp8(const void* gq, const void* gs, const void* xq,
                                   const void* xs, const int32_t* expert_off, int E, int M,
                                   int N, int K, size_t Mcap, void* out_bf16, int* status_dev,
                                   void* stream) {
  mgw_status st0 = wgrad_check(gq, gs, xq, xs, expert_off, E, M, N, K, Mcap, out_bf16);
  if (st0 != MGW_OK) return st0;
  DeviceInfo dev;
  mgw_status st = current_device(&dev);
  if (st != MGW_OK) return st;
  mgw::WgradArgs a;
  if (!wgrad_maps(&a, gq, gs, xq, xs, expert_off, E, M, N, K, Mcap, out_bf16, status_dev,
                  mgw::wgrad_uses_pair(E, N)))
    return MGW_ERR_CUDA;
#ifdef MGW_TEST_HOOKS
  {
    // Only in the test build of the library (libmgw_testhooks.so), see kernels.h.
    const char* v = std::getenv("MGW_TEST_DROP_LOAD");
    a.drop_first_load = (v != nullptr && v[0] == '1') ? 1 : 0;
  }
#endif
  const cudaError_t err = mgw::launch_grouped_wgrad(a, dev.sms, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MGW_OK : MGW_ERR_CUDA;
}

mgw_status mgw_grouped_dgrad_f32(const float* dy, const float* W, const int32_t* expert_off,
                                 int E, int rows, int out_f, int in_f, float* dx,
                                 int* status_dev, void* stream) {
  if (!W || !expert_off || (rows > 0 && (!dy || !dx))) return MGW_ERR_INVALID_ARG;
  if (rows < 0 || out_f <= 0 || in_f <= 0 || E < 1 || E > MGW_MAX_EXPERTS)
    return MGW_ERR_INVALID_ARG;
  if (out_f % 32 != 0 || in_f % 256 != 0) return MGW_ERR_UNSUPPORTED;
  // stacked weight rows e*out_f + n are TMA coordinates (32-bit)
  if (static_cast<long long>(E) * out_f >= (1ll << 31)) return MGW_ERR_UNSUPPORTED;
  if ((dy && !aligned16(dy)) || !aligned16(W) || (dx && !aligned16(dx)))
    return MGW_ERR_INVALID_ARG;
  DeviceInfo dev;
  mgw_status st = current_device(&dev);
  if (st != MGW_OK) return st;
  mgw::DgradArgs a;
  std::memset(&a, 0, sizeof(a));
  a.dy = dy;
  a.W = W;
  a.expert_off = expert_off;
  a.dx = dx;
  a.E = E;
  a.rows = rows;
  a.out_f = out_f;
  a.in_f = in_f;
  a.status = status_dev;
  a.dx_align32 = (reinterpret_cast<uintptr_t>(dx) & 31) == 0;
  // CTA pairs load 128 of a pair tile's 256 columns of W per CTA; the single-SM kernel 256
  const bool pair = mgw::dgrad_uses_pair(a, dev.sms);
  if (!make_map_2d(&a.tm_w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, W, in_f,
                   static_cast<uint64_t>(E) * out_f, static_cast<uint64_t>(in_f) * 4,
                   pair ? 128 : 256, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return MGW_ERR_CUDA;
  // dy rows by TMA, 128 rows x 32 columns per CTA and chunk (with no row there is no dy, and
  // the map, which the kernel then never reads, is made over W)
  if (!make_map_2d(&a.tm_dy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rows > 0 ? dy : W, out_f,
                   rows > 0 ? static_cast<uint64_t>(rows) : 1, static_cast<uint64_t>(out_f) * 4,
                   32, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return MGW_ERR_CUDA;
#ifdef MGW_TEST_HOOKS
  {
    // Only in the test build of the library (libmgw_testhooks.so), see kernels.h.
    const char* v = std::getenv("MGW_TEST_DROP_LOAD");
    a.drop_first_load = (v != nullptr && v[0] == '1') ? 1 : 0;
  }
#endif
  const cudaError_t err =
      pair ? mgw::launch_grouped_dgrad_pair(a, dev.sms, static_cast<cudaStream_t>(stream))
           : mgw::launch_grouped_dgrad(a, dev.sms, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MGW_OK : MGW_ERR_CUDA;
}

}  // extern "C"

namespace {

mgw_status grouped_mm_impl(const void* aq, const void* as, const void* bq, const void* bs,
                           const int32_t* expert_off, int E, int M, int J, int L, size_t Mcap,
                           uint64_t RB, uint64_t LB, long long b_row_step, long long b_col_step,
                           void* out_bf16, int* status_dev, void* stream) {
  DeviceInfo dev;
  mgw_status st = current_device(&dev);
  if (st != MGW_OK) return st;
  mgw::MmArgs a;
  std::memset(&a, 0, sizeof(a));
  // With M == 0 there is no routed row and the output map is never used.
  const void* out_base = M > 0 ? out_bf16 : aq;
  const uint64_t out_rows = M > 0 ? static_cast<uint64_t>(M) : 1;
  if (!make_map_2d(&a.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, aq, L, Mcap, L, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&a.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, bq, LB, RB, LB, 128, 256,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&a.tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out_base, J, out_rows,
                   static_cast<uint64_t>(J) * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return MGW_ERR_CUDA;
  a.out = out_bf16;
  a.as = static_cast<const uint8_t*>(as);
  a.bs = static_cast<const uint8_t*>(bs);
  a.expert_off = expert_off;
  a.E = E;
  a.M = M;
  a.J = J;
  a.L = L;
  a.Mcap = static_cast<long long>(Mcap);
  a.RB = static_cast<long long>(RB);
  a.b_row_step = b_row_step;
  a.b_col_step = b_col_step;
  a.status = status_dev;
  const cudaError_t err = mgw::launch_grouped_mm_mxfp8(a, dev.sms, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MGW_OK : MGW_ERR_CUDA;
}

}  // namespace

extern "C" {

mgw_status mgw_mxfp8_quantize_rows(const void* src_bf16, int src_rows, const int32_t* row_index,
                                   int M, int C, const int32_t* expert_off, int E, void* q_e4m3,
                                   void* scales_e8m0, size_t Mcap, int scale_rule,
                                   int* status_dev, void* stream) {
  if (!expert_off || !q_e4m3 || !scales_e8m0 || (M > 0 && !src_bf16)) return MGW_ERR_INVALID_ARG;
  if (M < 0 || C <= 0 || E < 1 || E > MGW_MAX_EXPERTS) return MGW_ERR_INVALID_ARG;
  if (scale_rule != MGW_SCALE_FLOOR && scale_rule != MGW_SCALE_CEIL_448) return MGW_ERR_INVALID_ARG;
  if (row_index != nullptr && M > 0 && src_rows < 1) return MGW_ERR_INVALID_ARG;
  if (C % 128 != 0) return MGW_ERR_UNSUPPORTED;
  if (Mcap % 128 != 0 || Mcap < mgw_mxfp8_token_capacity(M, E) || Mcap > (size_t(1) << 31))
    return MGW_ERR_CAPACITY;
  if ((src_bf16 && !aligned16(src_bf16)) || !aligned16(q_e4m3) || !aligned16(scales_e8m0))
    return MGW_ERR_INVALID_ARG;
  DeviceInfo dev;
  mgw_status st = current_device(&dev);
  if (st != MGW_OK) return st;
  const cudaError_t err = mgw::launch_mxfp8_quantize_rows(
      src_bf16, row_index != nullptr ? src_rows : M, row_index, M, C, expert_off, E, q_e4m3,
      scales_e8m0, static_cast<long long>(Mcap), scale_rule, status_dev, dev.sms,
      static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MGW_OK : MGW_ERR_CUDA;
}

mgw_status mgw_grouped_fprop_mxfp8(const void* xq, const void* xs, const void* wq,
                                   const void* ws, const int32_t* expert_off, int E, int M,
                                   int N, int K, size_t Mcap, size_t Mw, void* y_bf16,
                                   int* status_dev, void* stream) {
  if (!xq || !xs || !wq || !ws || !expert_off || (M > 0 && !y_bf16)) return MGW_ERR_INVALID_ARG;
  if (M < 0 || N <= 0 || K <= 0 || E < 1 || E > MGW_MAX_EXPERTS) return MGW_ERR_INVALID_ARG;
  if (N % 256 != 0 || K % 128 != 0) return MGW_ERR_UNSUPPORTED;
  if (Mcap % 128 != 0 || Mcap < mgw_mxfp8_token_capacity(M, E) || Mcap > (size_t(1) << 31))
    return MGW_ERR_CAPACITY;
  if (Mw % 128 != 0 || Mw < static_cast<size_t>(E) * N || Mw > (size_t(1) << 31))
    return MGW_ERR_CAPACITY;
  if (!aligned16(xq) || !aligned16(xs) || !aligned16(wq) || !aligned16(ws) ||
      (y_bf16 && !aligned16(y_bf16)))
    return MGW_ERR_INVALID_ARG;
  return grouped_mm_impl(xq, xs, wq, ws, expert_off, E, M, N, K, Mcap, Mw, K, N, 0, y_bf16,
                         status_dev, stream);
}

mgw_status mgw_grouped_dgrad_mxfp8(const void* dyq, const void* dys, const void* wtq,
                                   const void* wts, const int32_t* expert_off, int E, int M,
                                   int N, int K, size_t Mcap, size_t Mw, void* dx_bf16,
                                   int* status_dev, void* stream) {
  if (!dyq || !dys || !wtq || !wts || !expert_off || (M > 0 && !dx_bf16))
    return MGW_ERR_INVALID_ARG;
  if (M < 0 || N <= 0 || K <= 0 || E < 1 || E > MGW_MAX_EXPERTS) return MGW_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 256 != 0) return MGW_ERR_UNSUPPORTED;
  if (Mcap % 128 != 0 || Mcap < mgw_mxfp8_token_capacity(M, E) || Mcap > (size_t(1) << 31))
    return MGW_ERR_CAPACITY;
  if (Mw % 128 != 0 || Mw < static_cast<size_t>(E) * N || Mw > (size_t(1) << 31))
    return MGW_ERR_CAPACITY;
  if (!aligned16(dyq) || !aligned16(dys) || !aligned16(wtq) || !aligned16(wts) ||
      (dx_bf16 && !aligned16(dx_bf16)))
    return MGW_ERR_INVALID_ARG;
  return grouped_mm_impl(dyq, dys, wtq, wts, expert_off, E, M, K, N, Mcap, K, Mw, 0, N, dx_bf16,
                         status_dev, stream);
}

}  // extern "C"

#ifdef MGW_DIAG
extern "C" {

mgw_status mgw_diag_timeline(mgw_diag_record* out, int cap, int* total) {
  if (!total || cap < 0 || (cap > 0 && !out)) return MGW_ERR_INVALID_ARG;
  static_assert(sizeof(mgw_diag_record) == sizeof(mgw::DiagRecord), "record layout");
  using Read = cudaError_t (*)(mgw::DiagRecord*, int, int*);
  const Read readers[3] = {mgw::diag_timeline_read_wgrad, mgw::diag_timeline_read_dgrad,
                           mgw::diag_timeline_read_dgrad_pair};
  auto* dst = reinterpret_cast<mgw::DiagRecord*>(out);
  int copied = 0, recorded = 0;
  for (Read read : readers) {
    int n = 0;
    if (read(dst + copied, cap - copied, &n) != cudaSuccess) return MGW_ERR_CUDA;
    const int kept = n < mgw::kDiagTimelineCap ? n : mgw::kDiagTimelineCap;
    copied += kept < cap - copied ? kept : cap - copied;
    recorded += n;
  }
  *total = recorded;
  return MGW_OK;
}

mgw_status mgw_diag_timeline_reset(void) {
  if (mgw::diag_timeline_reset_wgrad() != cudaSuccess ||
      mgw::diag_timeline_reset_dgrad() != cudaSuccess ||
      mgw::diag_timeline_reset_dgrad_pair() != cudaSuccess)
    return MGW_ERR_CUDA;
  return MGW_OK;
}

}  // extern "C"
#endif  // MGW_DIAG
