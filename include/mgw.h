/*
 * mgw -- grouped MoE backward GEMMs for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libmgw.so.  Every entry point takes plain device pointers, sizes and
 * a CUDA stream handle; nothing here depends on PyTorch.  All device work is
 * asynchronous on `stream` (a cudaStream_t passed as void*; NULL means the
 * legacy default stream).  No entry point calls an allocator: the caller owns
 * every buffer it passes, and the one library-owned buffer is the static device
 * workspace of mgw_grouped_wgrad_mxfp8_balanced_noalloc.  Host-detectable
 * argument errors return a negative status before anything is launched; data
 * errors that only the device can see (an invalid expert_off array) are reported
 * by OR-ing MGW_DEV_* bits into the caller's int status word, and the kernels
 * then leave their outputs untouched.
 * No entry point aborts, traps or blocks the host.
 *
 * Limits common to every entry point: device pointers 16-byte aligned (else
 * MGW_ERR_INVALID_ARG); a padded token or row axis Mcap (or Mw) of at most 2^31
 * (else MGW_ERR_CAPACITY); 1 <= E <= MGW_MAX_EXPERTS.  The current device must be
 * compute capability 10.3 (else MGW_ERR_ARCH).
 *
 * Pages restated (cited by title and part):
 *   wgrad page  "tinygrad/extra/thunder/amd/grouped_mxfp8_wgrad.cpp" -- the
 *               grouped MXFP8 expert weight gradient kernel.
 *   dgrad page  "oarust grouped_gemm_m_data_backward.slang" -- the grouped fp32
 *               data-gradient compute shader.
 *   post-attn page  vLLM "models/minimax_m3/amd/mono/kernels/post_attn" -- its
 *               MXFP8 quantizer (mx8_scale / mx8_q) for the saturating clamp.
 *   OCP "OFP8 Formats" v1.0 and "Microscaling Formats (MX)" v1.0.
 */
#ifndef MGW_H
#define MGW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int mgw_status;

/* Return codes. */
#define MGW_OK 0
#define MGW_ERR_INVALID_ARG (-1)  /* null pointer, negative size, E out of range */
#define MGW_ERR_UNSUPPORTED (-2)  /* a size that is not a supported multiple */
#define MGW_ERR_CAPACITY (-3)     /* Mcap too small or not a multiple of 128 */
#define MGW_ERR_CUDA (-4)         /* a CUDA runtime/driver call or launch failed */
#define MGW_ERR_ARCH (-5)         /* current device is not compute capability 10.3 */

/* Bits OR-ed into *status_dev by the kernels (the caller zeroes it). */
#define MGW_DEV_BAD_OFFSETS 1 /* expert_off[0] != 0, decreasing, or expert_off[E] != M/rows */
#define MGW_DEV_TIMEOUT 2     /* an internal pipeline wait exceeded 1 s; outputs undefined */
#define MGW_DEV_BAD_INDEX 4   /* mgw_mxfp8_quantize_gather: a row index outside the source */
#define MGW_DEV_BOUNDS 8      /* diagnostic library only (mgw_diag.h): a computed address outside its tensor */

#define MGW_MAX_EXPERTS 1024

/* Scale rules of mgw_mxfp8_quantize. */
#define MGW_SCALE_FLOOR 0    /* OCP MX: 2^(floor(log2 amax) - 8), saturate to +-448 */
#define MGW_SCALE_CEIL_448 1 /* post-attn page's RoundUp: ceil_pow2(amax * fp32(1/448)) */

/* Human-readable name of a return code (static string). */
const char *mgw_status_string(mgw_status s);

/* Library version, major*10000 + minor*100 + patch. */
int mgw_version(void);

/* ------------------------------------------------------------- layout helpers
 * The quantized operands live on a padded token axis of length Mcap: expert e's
 * tokens start at P[e] = sum_{e'<e} ceil128(expert_off[e'+1] - expert_off[e']),
 * so every expert segment starts on a 128-token boundary and its tail up to the
 * next boundary is zero.  Host-only helpers, no device work. */

/* Smallest Mcap valid for any split of M tokens over E experts:
 * ceil128(M + 127*E).  Returns 0 for negative M or E < 1. */
size_t mgw_mxfp8_token_capacity(int M, int E);

/* Bytes of the e8m0 scale buffer for C features on an Mcap token axis: C*Mcap/32. */
size_t mgw_mxfp8_scale_bytes(int C, size_t Mcap);

/* --------------------------------------------------------------- quantize
 * mgw_mxfp8_quantize -- MXFP8 quantization of one wgrad operand along the token
 * (contraction) axis, transposed to token-contiguous rows.
 *
 * Defines the operands A = g^T and B = x^T of the wgrad page's kernel (its
 * `gl<fp8e4m3, 1, 1, N, M>` / `gl<fp8e4m3, 1, 1, K, M>` declarations and the
 * e8m0 scale tensors with four scales per 128 tokens).  For every feature c and
 * every block of 32 consecutive tokens of one expert (blocks restart at each
 * expert's first token and never mix experts):
 *   amax = max |v| over the block's tokens,
 *   scale = 2^s with, for scale_rule MGW_SCALE_FLOOR,
 *           s = clamp(floor(log2 amax) - 8, -127, 127)   (OCP MX rule; amax == 0 gives
 *           s = -127), or, for MGW_SCALE_CEIL_448 (the post-attn page's mx8_scale),
 *           s + 127 = clamp(biased exponent of ceil_pow2(amax * fp32(1/448)), 1, 254)
 *           with the product rounded to fp32 as that page computes it,
 *   q = e4m3(v / scale), rounded to nearest even, |q| saturated at 448 (the
 *       post-attn page's mx8_q clamp).
 * A 32-token block that holds no token of its expert (the padding up to the expert's
 * next 128-token boundary) gets scale byte 0 and values 0 under either rule.
 *
 * src_bf16   device, bf16 [M, C] row-major (token-major), read only.
 * M          tokens, >= 0.  C: features, a positive multiple of 128.
 * expert_off device int32 [E+1]: expert e owns tokens expert_off[e] ..
 *            expert_off[e+1]-1; must be 0 = off[0] <= off[1] <= ... <= off[E] = M.
 * E          experts, 1 .. MGW_MAX_EXPERTS.
 * q_e4m3     device, uint8 [C, Mcap]: row c holds feature c's e4m3 bytes on the
 *            padded token axis; every byte of the buffer is written (pads 0).
 * scales_e8m0 device, mgw_mxfp8_scale_bytes(C, Mcap) bytes, every byte written
 *            (pads 0), in tcgen05 scale-factor atoms: for feature c and padded
 *            token t the byte is at
 *              ((t/128) * (C/128) + c/128) * 512 + (c%32)*16 + ((c%128)/32)*4 + (t%128)/32.
 * Mcap       padded token axis, multiple of 128, >= mgw_mxfp8_token_capacity(M, E).
 * scale_rule MGW_SCALE_FLOOR or MGW_SCALE_CEIL_448; anything else is MGW_ERR_INVALID_ARG.
 * status_dev device int, nullable.  With NULL an invalid expert_off is not
 *            reported (the kernel still writes nothing).
 * Returns MGW_OK or a negative code; no work is launched on error.
 */
mgw_status mgw_mxfp8_quantize(const void *src_bf16, int M, int C, const int32_t *expert_off,
                              int E, void *q_e4m3, void *scales_e8m0, size_t Mcap,
                              int scale_rule, int *status_dev, void *stream);

/* mgw_mxfp8_quantize_gather -- the same quantization of the routed token matrix
 * x[t, :] = src[row_index[t], :] without materialising it.  In an MoE layer the routed
 * rows of one expert are copies of rows of the token (hidden-state) matrix; the
 * post-attn page's wide MoE path builds such per-expert row tables (its down_tables)
 * for the same gather.
 *
 * src_bf16   device, bf16 [src_rows, C] row-major (the unpermuted token matrix).
 * src_rows   rows of src, >= 1 when M > 0.
 * row_index  device int32 [M]: routed token t reads source row row_index[t].  An index
 *            outside [0, src_rows) is not read: that row is quantized as zeros and
 *            MGW_DEV_BAD_INDEX is set in *status_dev.
 * Every other argument, the output layout and the errors are those of
 * mgw_mxfp8_quantize. */
mgw_status mgw_mxfp8_quantize_gather(const void *src_bf16, int src_rows,
                                     const int32_t *row_index, int M, int C,
                                     const int32_t *expert_off, int E, void *q_e4m3,
                                     void *scales_e8m0, size_t Mcap, int scale_rule,
                                     int *status_dev, void *stream);

/* ---------------------------------------------------------------- wgrad
 * mgw_grouped_wgrad_mxfp8 -- grouped expert weight gradient
 *   grad_w[e*N + n, k] = sum over tokens t of expert e of g[t, n] * x[t, k]
 * from MXFP8 operands (each element times its block's e8m0 scale), accumulated
 * in fp32 and stored as bf16 (round to nearest even).  This is the wgrad page's
 * grouped_mxfp8_wgrad_kernel: per-expert token range from expert_off, scaled
 * fp8 MMAs over 32-token scale blocks, experts stacked along the output rows,
 * accumulators that start at zero so an expert without tokens gets zero rows.
 *
 * gq, gs     g quantized by mgw_mxfp8_quantize with C = N (same expert_off, Mcap).
 * xq, xs     x quantized by mgw_mxfp8_quantize with C = K.
 * expert_off device int32 [E+1], as for the quantizer; M = expert_off[E].
 * N          grad_w rows per expert, a positive multiple of 128.
 * K          grad_w columns, a positive multiple of 256.
 *            E*N <= 2^31 and E * (N/128) * (K/256) < 2^31 (output rows and tiles are
 *            counted in 32 bits); else MGW_ERR_UNSUPPORTED.
 * Mcap       the padded token axis both operands were quantized on.
 * out_bf16   device, bf16 [E*N, K] row-major, fully written.
 * status_dev device int, nullable (see MGW_DEV_*).
 * Gradients accumulate over at most 2^24 tokens per expert without loss of
 * fp32 integer-count exactness; inputs must be finite.
 */
mgw_status mgw_grouped_wgrad_mxfp8(const void *gq, const void *gs, const void *xq,
                                   const void *xs, const int32_t *expert_off, int E, int M,
                                   int N, int K, size_t Mcap, void *out_bf16, int *status_dev,
                                   void *stream);

/* -------------------------------------------------- wgrad under skewed routing
 * mgw_grouped_wgrad_mxfp8_balanced -- the same result as mgw_grouped_wgrad_mxfp8 (same
 * operands, layout, output and tolerance), computed with split-K over tokens and dynamic
 * scheduling for routings where a few experts hold most tokens.
 *
 * The wgrad page runs one block per (expert, output tile) over all of that expert's tokens
 * (its expert decode from the block index); with one huge expert a few blocks then carry
 * most of the work.  Here an expert whose 128-token chunks exceed a target item length L
 * (about all chunks / (2 x SM count), at least 8) is split into S = ceil(chunks / L) <= 16
 * token ranges per output tile; each range's fp32 partial goes to the workspace and the
 * range that finishes last sums the S partials in range order (so results are
 * deterministic) and stores bf16.  Items are handed out longest first by an atomic counter
 * in the workspace.  L is doubled until the partials fit the workspace; a workspace of
 * only the 256-byte header gives dynamic scheduling without splits.
 *
 * Arguments as mgw_grouped_wgrad_mxfp8, plus:
 * workspace        device, 256-byte aligned, workspace_bytes long, zero-filled before its
 *                  first use.  Every call that ends without MGW_DEV_TIMEOUT returns its
 *                  counters (the first 256 + 4 x slots bytes) to zero, so it is reused as
 *                  is; after a time-out it must be zero-filled again.  Calls sharing a
 *                  workspace must not run concurrently.
 * workspace_bytes  >= 256 (else MGW_ERR_CAPACITY); mgw_grouped_wgrad_workspace_bytes gives
 *                  a size with room for 2 x SM count partial tiles (128 KB each).
 * E <= 512 (else MGW_ERR_UNSUPPORTED). */
mgw_status mgw_grouped_wgrad_mxfp8_balanced(const void *gq, const void *gs, const void *xq,
                                            const void *xs, const int32_t *expert_off, int E,
                                            int M, int N, int K, size_t Mcap, void *out_bf16,
                                            void *workspace, size_t workspace_bytes,
                                            int *status_dev, void *stream);

/* mgw_grouped_wgrad_mxfp8_balanced_noalloc -- mgw_grouped_wgrad_mxfp8_balanced for callers
 * that cannot allocate device memory: code running inside a memory pool or an allocator
 * that must not be re-entered, a captured graph's fixed memory plan, or an embedding that
 * owns every allocation of the process.  The pages have no counterpart to this entry point;
 * it exists for those callers only.
 *
 * The workspace is owned by the library: a 16 MB device array (the counters plus room for
 * 128 fp32 partial tiles of 128 x 256) defined in the library, zero-filled when the library
 * loads, held by every GPU that loads it until the process exits.  The call allocates and
 * frees nothing (no cudaMalloc, no cudaFree, no allocating library routine).  Its device
 * address is looked up with cudaGetSymbolAddress on the first call in each CUDA context
 * (again after the context is re-created), so make that first call before any stream
 * capture.  Every call first clears the array's counters (under 1 KB, cudaMemsetAsync on
 * `stream`), so a call after one that ended with MGW_DEV_TIMEOUT starts clean.  Every call
 * on a device shares the one array: calls whose work overlaps on the GPU (different
 * streams, or several host threads) race and give undefined results.
 *
 * The 128 partial slots bound the split-K: splits apply only while the split tiles'
 * partials, sum over split experts of (N/128)*(K/256)*S, fit in 128; otherwise the target
 * item length doubles until they do, and with more than 64 output tiles per expert no
 * expert is split (every call still gets the longest-first dynamic scheduling).  No size
 * is rejected for the workspace's sake.  Arguments, result, limits (E <= 512) and errors
 * otherwise as mgw_grouped_wgrad_mxfp8_balanced. */
mgw_status mgw_grouped_wgrad_mxfp8_balanced_noalloc(const void *gq, const void *gs,
                                                    const void *xq, const void *xs,
                                                    const int32_t *expert_off, int E, int M,
                                                    int N, int K, size_t Mcap, void *out_bf16,
                                                    int *status_dev, void *stream);

/* Workspace size for mgw_grouped_wgrad_mxfp8_balanced on the current device: 2 x SM count
 * partial tiles plus counters (about 38 MB on a 152-SM GB300).  0 if no usable device. */
size_t mgw_grouped_wgrad_workspace_bytes(int E, int N, int K);

/* ---------------------------------------------------------------- dgrad
 * mgw_grouped_dgrad_f32 -- grouped data gradient
 *   dx[r, k] = sum_n dy[r, n] * W[e(r), n, k]
 * where e(r) is the expert whose row range expert_off[e] <= r < expert_off[e+1]
 * holds r (the dgrad page's expert_for_row; empty experts own no row).  fp32
 * in and out, computed with 3xTF32 tensor-core products (hi*hi + hi*lo + lo*hi,
 * Ootomo & Yokota 2022) and fp32 accumulation.  Row segments need not align to
 * any tile.
 *
 * dy         device, fp32 [rows, out_f] row-major.
 * W          device, fp32 [E, out_f, in_f] row-major (in_f contiguous), the dgrad
 *            page's weight layout W[(e*out_f + n)*in_f + k].
 * expert_off device int32 [E+1], 0 = off[0] <= ... <= off[E] = rows.
 * rows >= 0; out_f a positive multiple of 32; in_f a positive multiple of 256;
 * E * out_f < 2^31 (the stacked weight rows are addressed with 32-bit
 * coordinates; else MGW_ERR_UNSUPPORTED).
 * dx         device, fp32 [rows, in_f] row-major, fully written.
 * status_dev device int, nullable.
 */
mgw_status mgw_grouped_dgrad_f32(const float *dy, const float *W, const int32_t *expert_off,
                                 int E, int rows, int out_f, int in_f, float *dx,
                                 int *status_dev, void *stream);

/* ---------------------------------------- forward and data gradient in MXFP8
 * The expert GEMMs on routed rows with both operands MXFP8 along the contraction
 * axis, as the post-attn page runs its expert GEMMs on MXFP8 activations and
 * weights (one e8m0 byte per 32 hidden features of a token row; its wide MoE up
 * and down stages).  Routed rows of expert e are expert_off[e] <= r <
 * expert_off[e+1]; row-wise quantized operands hold them on a padded row axis of
 * length Mcap, expert e's rows from P[e] (the padded starts above), so every
 * 128-row tile belongs to one expert. */

/* mgw_mxfp8_quantize_rows -- row-wise MXFP8 quantization (no transpose).
 * For every routed row r of expert e and every block of 32 consecutive columns:
 * the scale byte from the block's largest magnitude under scale_rule (as
 * mgw_mxfp8_quantize), values scaled by the power of two and rounded to e4m3
 * (nearest even, saturating to +-448), written to padded row P[e] + (r - off[e]).
 *
 * src_bf16    device, bf16 [src_rows, C] row-major (C contiguous).
 * src_rows    rows of src when row_index is given; ignored otherwise.
 * row_index   device int32 [M], nullable.  When given, routed row r reads row
 *             row_index[r] of src (the unpermuted token matrix: the MoE gather);
 *             an index outside [0, src_rows) gives a zero row and sets
 *             MGW_DEV_BAD_INDEX.  When null, routed row r is row r of src [M, C].
 * M           routed rows (>= 0); C a positive multiple of 128.
 * expert_off  device int32 [E+1], 0 = off[0] <= ... <= off[E] = M.
 * q_e4m3      device, [Mcap, C] row-major e4m3 bytes, fully written (padding rows 0).
 * scales_e8m0 device, Mcap*C/32 bytes, fully written: 512-byte atoms, the atom of
 *             128-column chunk c and 128-row tile t at byte (c*(Mcap/128) + t)*512,
 *             row p%128 = r0 + 32*r1 and 32-column block kb of the chunk at
 *             16*r0 + 4*r1 + kb (the layout mgw_mxfp8_quantize writes for a
 *             [C, Mcap] operand, here for an [Mcap, C] one).  Padding bytes 0.
 * Mcap        multiple of 128, >= mgw_mxfp8_token_capacity(M, E).
 * All pointers 16-byte aligned.  Bad offsets: MGW_DEV_BAD_OFFSETS, outputs untouched. */
mgw_status mgw_mxfp8_quantize_rows(const void *src_bf16, int src_rows, const int32_t *row_index,
                                   int M, int C, const int32_t *expert_off, int E, void *q_e4m3,
                                   void *scales_e8m0, size_t Mcap, int scale_rule,
                                   int *status_dev, void *stream);

/* mgw_grouped_fprop_mxfp8 -- grouped forward GEMM
 *   y[r, n] = sum_k deq(x)[r, k] * deq(W)[e(r), n, k]
 * xq, xs   x quantized by mgw_mxfp8_quantize_rows with expert_off: [Mcap, K].
 * wq, ws   W [E, N, K] (bf16, nn.Linear layout) quantized by mgw_mxfp8_quantize_rows as
 *          [E*N, K] with offsets {0, N, 2N, ..., E*N} (W[e][n] is row e*N + n):
 *          [Mw, K] with Mw its Mcap.
 * N a positive multiple of 256; K a positive multiple of 128.
 * Mw a multiple of 128 and >= E*N (else MGW_ERR_CAPACITY).
 * y_bf16   device, bf16 [M, N] row-major, fully written (round to nearest even).
 * Accumulation is fp32 in tensor memory; no bound beyond fp32 summation error. */
mgw_status mgw_grouped_fprop_mxfp8(const void *xq, const void *xs, const void *wq,
                                   const void *ws, const int32_t *expert_off, int E, int M,
                                   int N, int K, size_t Mcap, size_t Mw, void *y_bf16,
                                   int *status_dev, void *stream);

/* mgw_grouped_dgrad_mxfp8 -- grouped data gradient with MXFP8 operands
 *   dx[r, k] = sum_n deq(dy)[r, n] * deq(W)[e(r), n, k]
 * (the dgrad page's product, contracted over the expert's output features n).
 * dyq, dys dy [M, N] quantized by mgw_mxfp8_quantize_rows with expert_off: [Mcap, N].
 * wtq, wts W [E, N, K] (bf16) quantized along n by mgw_mxfp8_quantize as [E*N, K]
 *          tokens-by-features with offsets {0, N, ..., E*N}: [K, Mw] with Mw its Mcap,
 *          W[e][n][k] at row k, column e*N + n.
 * N a positive multiple of 128; K a positive multiple of 256.
 * Mw a multiple of 128 and >= E*N (else MGW_ERR_CAPACITY).
 * dx_bf16  device, bf16 [M, K] row-major, fully written. */
mgw_status mgw_grouped_dgrad_mxfp8(const void *dyq, const void *dys, const void *wtq,
                                   const void *wts, const int32_t *expert_off, int E, int M,
                                   int N, int K, size_t Mcap, size_t Mw, void *dx_bf16,
                                   int *status_dev, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MGW_H */
