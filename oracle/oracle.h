/*
 * Plain CPU oracle for the grouped MoE backward GEMMs (MXFP8 wgrad, fp32 dgrad,
 * MXFP8 quantization).  TEST INFRASTRUCTURE ONLY: nothing on the product path
 * may include, link or call this code.  It shares no source with the CUDA
 * library; it is slow on purpose, fp64 throughout, with no blocking, fusion or
 * reordering beyond the plain definitions.
 *
 * Sources (page titles as cited in the docstrings below):
 *   [wgrad page]  tinygrad/extra/thunder/amd/grouped_mxfp8_wgrad.cpp
 *   [dgrad page]  oarust grouped_gemm_m_data_backward.slang
 *   [post-attn page] vLLM MiniMax-M3 AMD post_attn kernels (quantization rule)
 *   OCP "OFP8 Formats" v1.0 and OCP "Microscaling Formats (MX)" v1.0.
 *
 * Every function here is pinned by tests in tests/test_oracle_*.py against
 * values fixed by the pages or by mathematics; none is "parity unpinned".
 */
#ifndef MGW_ORACLE_H
#define MGW_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* OCP OFP8 E4M3: value of one byte (NaN for S.1111.111). */
double orc_e4m3_decode(uint8_t b);
/* OCP OFP8 E4M3: round-to-nearest-even of v, saturating |v| beyond 448 to 448. */
uint8_t orc_e4m3_encode_rne_satfinite(double v);
/* OCP MX E8M0: 2^(b-127); NaN for 255. */
double orc_e8m0_decode(uint8_t b);
/* MX shared-exponent rule for one block: byte of 2^(floor(log2 amax) - 8),
 * clamped to [-127, 127] before the +127 bias; amax == 0 gives byte 0. */
uint8_t orc_mx_scale_byte(double amax);
/* The post-attn page's RoundUp rule (its mx8_scale): byte = biased exponent of
 * ceil_pow2(amax * fp32(1/448)), the product taken in fp32 as the page does, clamped to
 * [1, 254].  Values are then scaled by 2^(127-byte) and clamped to +-448 (its mx8_q). */
uint8_t orc_mx_scale_byte_ceil448(double amax);
/* bf16 bit pattern -> exact value. */
double orc_bf16_decode(uint16_t h);

/* 128-padded start of each expert's token segment in the quantized layout:
 * P[0] = 0, P[e+1] = P[e] + ceil128(off[e+1] - off[e]).  Writes E+1 entries. */
void orc_padded_starts(const int32_t *off, int E, int64_t *P);

/* MXFP8 quantization of a bf16 [M, C] row-major matrix along the token axis,
 * blocks of 32 tokens restarting at each expert's first token.
 *   q  : [C, Mcap] e4m3 bytes, token-contiguous, expert e at P[e]; pads 0.
 *   sc : [C, Mcap/32] e8m0 bytes (plain layout), block j of expert e at
 *        P[e]/32 + j; pads 0. */
/* rule 0: the MX floor rule (orc_mx_scale_byte); rule 1: the RoundUp rule
 * (orc_mx_scale_byte_ceil448). */
void orc_mxfp8_quantize(const uint16_t *src, int M, int C, const int32_t *off, int E,
                        int64_t Mcap, int rule, uint8_t *q, uint8_t *sc);

/* Grouped wgrad: out[(e*N+n)*K + k] = sum_{t<cnt_e} deq(g)[n, P_e+t] * deq(x)[k, P_e+t]
 * in fp64, from the quantized operands (q and plain scales as above). */
void orc_grouped_wgrad(const uint8_t *gq, const uint8_t *gs, const uint8_t *xq,
                       const uint8_t *xs, const int32_t *off, int E, int N, int K,
                       int64_t Mcap, double *out);
/* One element of the same (for sampled checks at full size). */
double orc_grouped_wgrad_element(const uint8_t *gq, const uint8_t *gs, const uint8_t *xq,
                                 const uint8_t *xs, const int32_t *off, int E, int64_t Mcap,
                                 int e, int n, int k);

/* Row -> expert rule of the dgrad page (linear scan over offsets[1..E-1]). */
int orc_expert_for_row_scan(const int32_t *off, int E, int row);
/* Same rule by binary search: the last e in [0, E) with off[e] <= row, taking the
 * largest such e (so empty experts are skipped). */
int orc_expert_for_row_bsearch(const int32_t *off, int E, int row);

/* Grouped dgrad: dx[r,k] = sum_n dy[r,n] * W[e(r), n, k] in fp64, and
 * bound[r,k] = sum_n |dy[r,n]| * |W[e(r),n,k]|.  bound may be NULL. */
void orc_grouped_dgrad(const float *dy, const float *W, const int32_t *off, int E, int rows,
                       int out_f, int in_f, double *dx, double *bound);
/* One element of the same; *bound_out may be NULL. */
double orc_grouped_dgrad_element(const float *dy, const float *W, const int32_t *off, int E,
                                 int rows, int out_f, int in_f, int r, int k, double *bound_out);

/* The dgrad page's fp32 formulation (32-row groups; a group within one expert takes
 * that expert's weights, a straddling group looks up each row; running fp32 sums over
 * n in order, fused multiply-add when fused != 0).  A cross-check of orc_grouped_dgrad,
 * which any correct result must match within 1e-5 * bound. */
void orc_grouped_dgrad_page_f32(const float *dy, const float *W, const int32_t *off, int E,
                                int rows, int out_f, int in_f, int fused, float *dx);

/* ----------------------------------------------- forward and data-gradient GEMMs
 * MXFP8 operands quantized along the hidden (contraction) axis of each row. */

/* Row-wise MXFP8 quantization of a bf16 [M, C] row-major matrix: one scale per 32
 * consecutive elements of a row (blocks along C, starting at column 0), rows of
 * expert e placed at the padded rows P[e] + (r - off[e]).
 *   q  : [Mcap, C] e4m3 bytes, row-major; padding rows 0.
 *   sc : [Mcap, C/32] e8m0 bytes (plain layout); padding 0.
 * rule as in orc_mxfp8_quantize. */
void orc_mxfp8_quantize_rows(const uint16_t *src, int M, int C, const int32_t *off, int E,
                             int64_t Mcap, int rule, uint8_t *q, uint8_t *sc);

/* sum_l deq(a)[l] * deq(b)[l] over L elements (L % 32 == 0), one e8m0 scale per 32. */
double orc_mx_dot(const uint8_t *aq, const uint8_t *as, const uint8_t *bq, const uint8_t *bs,
                  int L);

/* Grouped forward GEMM y[r, n] = sum_k deq(x)[r, k] * deq(W)[e(r), n, k] in fp64.
 *   xq, xs : row-wise quantized x ([Mcap, K], plain scales [Mcap, K/32]), rows by off.
 *   wq, ws : row-wise quantized W stacked [Mw, K] (plain scales [Mw, K/32]); W[e][n]
 *            is row Pw[e] + n, Pw the padded starts of w_off (E+1 entries, e*N).
 *   out    : [M, N]. */
void orc_grouped_fprop_mx(const uint8_t *xq, const uint8_t *xs, const uint8_t *wq,
                          const uint8_t *ws, const int32_t *off, const int32_t *w_off, int E,
                          int M, int N, int K, int64_t Mcap, double *out);

/* Grouped data gradient dx[r, k] = sum_n deq(dy)[r, n] * deq(W)[e(r), n, k] in fp64.
 *   dyq, dys : row-wise quantized dy ([Mcap, N], plain scales [Mcap, N/32]), rows by off.
 *   wtq, wts : W quantized along n per expert (orc_mxfp8_quantize of W stacked
 *              [E*N, K] with w_off): [K, Mw] and plain scales [K, Mw/32]; W[e][n][k] is
 *              column Pw[e] + n of row k.
 *   out      : [M, K]. */
void orc_grouped_dgrad_mx(const uint8_t *dyq, const uint8_t *dys, const uint8_t *wtq,
                          const uint8_t *wts, const int32_t *off, const int32_t *w_off, int E,
                          int M, int N, int K, int64_t Mcap, int64_t Mw, double *out);

#ifdef __cplusplus
}
#endif
#endif
