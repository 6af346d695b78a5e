// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mgw {

constexpr int kMaxExperts = 1024;
// Experts the CTA-pair wgrad kernel takes (its expert tables share shared memory with a
// six-stage ring); more experts, or N % 256 != 0, use the single-SM kernel.
constexpr int kMaxPairExperts = 512;

size_t quantize_smem_bytes(int E);
// tm_src: bf16 [M, C] source, box 128 features x 128 tokens, no swizzle.
// tm_q:   e4m3 [C, Mcap] destination, box 128 tokens x 128 features, 128B swizzle.
// With row_index != nullptr the source rows are gathered: token t reads row
// row_index[t] of gsrc [src_rows, C] (tm_src is then unused).
cudaError_t launch_mxfp8_quantize(const CUtensorMap& tm_src, const CUtensorMap& tm_q, int M,
                                  int C, const int32_t* expert_off, int E, void* sc,
                                  long long Mcap, int rule, int* status, int num_sms,
                                  cudaStream_t stream, const void* gsrc = nullptr,
                                  const int32_t* row_index = nullptr, int src_rows = 0);

// Unique id of the calling thread's current CUDA context, or 0 when there is none yet.
// Unlike a context handle it is never reused within the process, so per-context state
// (kernel attributes, module symbol addresses) keyed on it is set up again for a context
// that was destroyed and re-created (cudaDeviceReset).
uint64_t current_context_id();

// Sets the kernel's maximum dynamic shared memory once per context and calling thread.
cudaError_t set_smem_attr_once(const void* kernel, size_t bytes, uint64_t* done_ctx);

// True when the static wgrad runs on CTA pairs (tcgen05 cta_group::2): then tm_b's box
// is 128 rows (each CTA holds half of the 256-column tile) and tm_sfa / tm_sfb are used.
bool wgrad_uses_pair(int E, int N);

struct WgradArgs {
  CUtensorMap tm_a;    // g^T e4m3 [N, Mcap], box 128 tokens x 128 rows, 128B swizzle
  CUtensorMap tm_b;    // x^T e4m3 [K, Mcap], box 128 tokens x 256 rows (128 for pairs), 128B swizzle
  CUtensorMap tm_sfa;  // CTA pairs: g scale atoms as 256-byte rows, box 256 x 2 (one atom)
  CUtensorMap tm_sfb;  // CTA pairs: x scale atoms as 256-byte rows, box 256 x 4 (two atoms)
  CUtensorMap tm_out;  // grad_w bf16 [E*N, K], box 64 cols x 128 rows, 128B swizzle
  void* out;           // grad_w (plain stores of the zero tiles)
  const uint8_t* gs;   // g scale atoms
  const uint8_t* xs;   // x scale atoms
  const int32_t* expert_off;
  int E, M, N, K;
  long long mcap;      // token capacity of the quantized operands (bounds checks of the diag build)
  int* status;
  // Test hook for the device time limit: when set, the static kernel's producer announces
  // its first chunk's bytes but never issues the copies, so the waits on that stage run out
  // and the kernel reports MGW_DEV_TIMEOUT.  Always zero in libmgw.so; only the test build
  // libmgw_testhooks.so (compiled with MGW_TEST_HOOKS) sets it, from MGW_TEST_DROP_LOAD=1.
  int drop_first_load;
  // Load-balanced kernel only (wgrad_balanced.cu): the workspace.
  int* ws_sched;   // [0] next item, [1] CTAs finished (zero at rest)
  int* ws_cnt;     // per split tile: parts finished (zero at rest), ws_slots entries
  float* ws_part;  // ws_slots fp32 128 x 256 partial tiles
  int ws_slots;
};
cudaError_t launch_grouped_wgrad(const WgradArgs& a, int num_sms, cudaStream_t stream);

// Load-balanced wgrad (wgrad_balanced.cu).  Workspace: a 256-byte header (item and CTA
// counters), ws_slots int tile counters (padded to 256 bytes), then ws_slots 128 KB fp32
// partial tiles.  Zero-filled before the first call; every call that ends without a
// device time-out leaves it zero-filled again.
constexpr int kMaxBalancedExperts = 512;
constexpr size_t kWsHeaderBytes = 256;
int balanced_workspace_slots(size_t bytes);   // -1 when smaller than the header
size_t balanced_workspace_bytes(int slots);
cudaError_t launch_grouped_wgrad_balanced(WgradArgs a, void* workspace, int slots, int num_sms,
                                          cudaStream_t stream);
// The library-owned workspace of the no-allocation entry point (wgrad_noalloc.cu): its
// device address in the current context, its size, and the size of its leading counter
// region (header and tile counters), which each call clears before it launches.
cudaError_t noalloc_wgrad_workspace(void** ptr, size_t* bytes, size_t* counter_bytes);

// Row-wise MXFP8 quantization (quantize_rows.cu): routed row r (source row row_index[r],
// or r when row_index is null) of expert e goes to padded row P[e] + r - off[e] of
// q [Mcap, C]; scale atoms per (128-column chunk, 128-row tile).
size_t quantize_rows_smem_bytes(int E);
cudaError_t launch_mxfp8_quantize_rows(const void* src, int src_rows, const int32_t* row_index,
                                       int M, int C, const int32_t* expert_off, int E, void* q,
                                       void* sc, long long Mcap, int rule, int* status,
                                       int num_sms, cudaStream_t stream);

// M-grouped MXFP8 GEMM (grouped_mm.cu): out[r, j] = sum_l A[p(r), l] * B[e*b_row_step + j,
// e*b_col_step + l], r a routed row of expert e, p(r) its padded row.
struct MmArgs {
  CUtensorMap tm_a;    // A e4m3 [Mcap, L], box 128 x 128 rows, 128B swizzle
  CUtensorMap tm_b;    // B e4m3 [RB, LB], box 128 x 256 rows, 128B swizzle
  CUtensorMap tm_out;  // out bf16 [M, J], box 64 cols x 128 rows, 128B swizzle
  void* out;           // out (plain stores of tiles that end inside an expert's last rows)
  const uint8_t* as;   // A scale atoms, (chunk * Mcap/128 + row tile) * 512
  const uint8_t* bs;   // B scale atoms, (chunk * RB/128 + row tile) * 512
  const int32_t* expert_off;
  int E, M, J, L;
  long long Mcap, RB;
  long long b_row_step, b_col_step;
  int* status;
};
cudaError_t launch_grouped_mm_mxfp8(const MmArgs& a, int num_sms, cudaStream_t stream);

struct DgradArgs {
  CUtensorMap tm_w;    // W fp32 [E*out_f, in_f], box 256 columns x 32 rows, no swizzle
  CUtensorMap tm_dy;   // dy fp32 [rows, out_f], box 32 columns x 128 rows, 128B swizzle
  const float* dy;
  const float* W;
  const int32_t* expert_off;
  float* dx;
  int E, rows, out_f, in_f;
  int* status;
  int dx_align32;      // dx is 32-byte aligned: the epilogue stores whole 32-byte sectors
  // Test hook for the device time limit, as in WgradArgs: the producer announces its first
  // raw stage's bytes but never issues the copies.  Only libmgw_testhooks.so sets it.
  int drop_first_load;
};
cudaError_t launch_grouped_dgrad(const DgradArgs& a, int num_sms, cudaStream_t stream);

// CTA-pair dgrad (dgrad_pair.cu): pair tiles of 256 rows x 256 columns, for problems with
// enough of them to keep the SM pairs busy; tm_w's box is then 128 columns x 32 rows.
bool dgrad_uses_pair(const DgradArgs& a, int num_sms);
cudaError_t launch_grouped_dgrad_pair(const DgradArgs& a, int num_sms, cudaStream_t stream);

// Work-item timeline of the diagnostic library (libmgw_diag.so, compiled with MGW_DIAG): one
// record per CTA and work item, the layout of mgw_diag_record in include/mgw_diag.h.
struct DiagRecord {
  uint32_t kernel, sm, cta, pad;
  long long item;
  uint64_t t_wait, t_done;
};
constexpr int kDiagTimelineCap = 65536;  // records kept per kernel family
#ifdef MGW_DIAG
cudaError_t diag_timeline_read_wgrad(DiagRecord* host, int cap, int* count);
cudaError_t diag_timeline_reset_wgrad();
cudaError_t diag_timeline_read_dgrad(DiagRecord* host, int cap, int* count);
cudaError_t diag_timeline_reset_dgrad();
cudaError_t diag_timeline_read_dgrad_pair(DiagRecord* host, int cap, int* count);
cudaError_t diag_timeline_reset_dgrad_pair();
#endif

}  // namespace mgw
