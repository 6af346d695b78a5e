/*
 * Plain fp64 CPU oracle -- TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Written from the definitions, not tuned: triple loops, fp64 sums, no blocking.
 * Only tests/, the smoke check and the benchmark's CPU-baseline leg use it.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- formats */

/* OCP OFP8 v1.0, E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 encodes subnormals m * 2^-9; S.1111.111 is NaN; there are no
 * infinities, so the largest finite magnitude is 1.75 * 2^8 = 448 (0x7E). */
double orc_e4m3_decode(uint8_t b) {
  const int sign = b >> 7;
  const int ex = (b >> 3) & 0xF;
  const int man = b & 0x7;
  if (ex == 0xF && man == 0x7) return NAN;
  double mag;
  if (ex == 0)
    mag = ldexp((double)man, -9);            /* 0.mmm * 2^(1-7) */
  else
    mag = ldexp(8.0 + (double)man, ex - 10); /* 1.mmm * 2^(ex-7) */
  return sign ? -mag : mag;
}

/* Round to nearest, ties to even, then saturate to the largest finite value.
 * The non-negative finite codes 0x00..0x7E are strictly increasing in value,
 * so the two neighbours of |v| are found by bisection over the codes, and
 * "even" means the code whose last mantissa bit (its last bit) is 0. */
uint8_t orc_e4m3_encode_rne_satfinite(double v) {
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs(v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 0x7E; /* invariant: dec(lo) <= a < dec(hi) */
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (orc_e4m3_decode((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid;
  }
  const double dlo = a - orc_e4m3_decode((uint8_t)lo);
  const double dhi = orc_e4m3_decode((uint8_t)hi) - a;
  int code;
  if (dlo < dhi)
    code = lo;
  else if (dhi < dlo)
    code = hi;
  else
    code = (lo % 2 == 0) ? lo : hi;
  return (uint8_t)(sign | code);
}

/* OCP MX v1.0, E8M0: an unsigned biased exponent, value 2^(b-127); 0xFF is NaN. */
double orc_e8m0_decode(uint8_t b) {
  if (b == 0xFF) return NAN;
  return ldexp(1.0, (int)b - 127);
}

/* OCP MX v1.0 shared exponent for an element format whose largest power of two
 * is 2^8 (E4M3): X = floor(log2(amax)) - 8, kept within the E8M0 range
 * [-127, 127].  floor(log2) comes from frexp, which is exact. */
uint8_t orc_mx_scale_byte(double amax) {
  if (amax == 0.0) return 0; /* empty block: scale 2^-127, values all zero */
  int ex = 0;
  (void)frexp(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1) */
  int s = (ex - 1) - 8;
  if (s < -127) s = -127;
  if (s > 127) s = 127;
  return (uint8_t)(s + 127);
}

/* The post-attn page's mx8_scale: amax times the fp32 constant 1/448, rounded to fp32;
 * the biased exponent of that product, plus one when its mantissa is not zero (rounding
 * up to a power of two); kept within [1, 254]. */
uint8_t orc_mx_scale_byte_ceil448(double amax) {
  const float r = (float)amax * (1.0f / 448.0f);
  uint32_t bits;
  memcpy(&bits, &r, sizeof bits);
  int e = (int)((bits >> 23) & 0xFFu);
  if ((bits & 0x7FFFFFu) != 0) e += 1;
  if (e > 254) e = 254;
  if (e < 1) e = 1;
  return (uint8_t)e;
}

double orc_bf16_decode(uint16_t h) {
  /* bf16 is the top half of an IEEE binary32; widen by placing it there. */
  const uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------- layout map */

static int64_t ceil128(int64_t v) { return (v + 127) / 128 * 128; }

void orc_padded_starts(const int32_t *off, int E, int64_t *P) {
  P[0] = 0;
  for (int e = 0; e < E; ++e) P[e + 1] = P[e] + ceil128((int64_t)off[e + 1] - off[e]);
}

/* ---------------------------------------------------------------- quantize */

/* Quantization of the wgrad operands.  The wgrad page takes g^T and x^T already
 * in e4m3 with one e8m0 scale per 32 tokens along the token (contraction) axis
 * (kernel arguments A, B, scale_A, scale_B and the `gl` declarations at its top).
 * The scale rule is the MX one, 2^(floor(log2 amax) - 8); values beyond the
 * e4m3 range after scaling are clamped to +-448 as the post-attn page's mx8_q
 * does, and rounding is to nearest even.  Blocks start at each expert's first
 * token, so no block mixes two experts.  With rule 1 the scale follows that page's
 * RoundUp rule instead. */
void orc_mxfp8_quantize(const uint16_t *src, int M, int C, const int32_t *off, int E,
                        int64_t Mcap, int rule, uint8_t *q, uint8_t *sc) {
  (void)M;
  const int64_t nsc = Mcap / 32;
  memset(q, 0, (size_t)C * (size_t)Mcap);
  memset(sc, 0, (size_t)C * (size_t)nsc);
  int64_t *P = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
  orc_padded_starts(off, E, P);
  for (int e = 0; e < E; ++e) {
    const int t0 = off[e];
    const int cnt = off[e + 1] - off[e];
    const int nblk = (cnt + 31) / 32;
    for (int c = 0; c < C; ++c) {
      for (int j = 0; j < nblk; ++j) {
        const int b0 = 32 * j;
        const int b1 = (b0 + 32 < cnt) ? b0 + 32 : cnt;
        double amax = 0.0;
        for (int t = b0; t < b1; ++t) {
          const double v = fabs(orc_bf16_decode(src[(int64_t)(t0 + t) * C + c]));
          if (v > amax) amax = v;
        }
        const uint8_t byte = rule ? orc_mx_scale_byte_ceil448(amax) : orc_mx_scale_byte(amax);
        const int s = (int)byte - 127;
        sc[(int64_t)c * nsc + P[e] / 32 + j] = byte;
        for (int t = b0; t < b1; ++t) {
          const double v = orc_bf16_decode(src[(int64_t)(t0 + t) * C + c]);
          q[(int64_t)c * Mcap + P[e] + t] = orc_e4m3_encode_rne_satfinite(ldexp(v, -s));
        }
      }
    }
  }
  free(P);
}

/* ------------------------------------------------------------------- wgrad */

static double deq(const uint8_t *q, const uint8_t *s, int64_t Mcap, int row, int64_t t) {
  return orc_e4m3_decode(q[(int64_t)row * Mcap + t]) *
         orc_e8m0_decode(s[(int64_t)row * (Mcap / 32) + t / 32]);
}

/* The wgrad page's kernel: for expert e, grad_w rows e*N .. e*N+N-1 hold
 * g_e^T x_e, contracted over the tokens expert_off[e] .. expert_off[e+1]-1
 * (its expert decode from the block index and its stacked-output store), with
 * accumulators that start at zero, so an expert without tokens stores zeros. */
void orc_grouped_wgrad(const uint8_t *gq, const uint8_t *gs, const uint8_t *xq,
                       const uint8_t *xs, const int32_t *off, int E, int N, int K,
                       int64_t Mcap, double *out) {
  int64_t *P = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
  orc_padded_starts(off, E, P);
  for (int e = 0; e < E; ++e) {
    const int cnt = off[e + 1] - off[e];
    /* dequantize the expert's slice once: gd[n][t], xd[k][t] */
    double *gd = (double *)malloc(sizeof(double) * (size_t)N * (size_t)(cnt > 0 ? cnt : 1));
    double *xd = (double *)malloc(sizeof(double) * (size_t)K * (size_t)(cnt > 0 ? cnt : 1));
    for (int n = 0; n < N; ++n)
      for (int t = 0; t < cnt; ++t) gd[(int64_t)n * cnt + t] = deq(gq, gs, Mcap, n, P[e] + t);
    for (int k = 0; k < K; ++k)
      for (int t = 0; t < cnt; ++t) xd[(int64_t)k * cnt + t] = deq(xq, xs, Mcap, k, P[e] + t);
    for (int n = 0; n < N; ++n)
      for (int k = 0; k < K; ++k) {
        double acc = 0.0;
        for (int t = 0; t < cnt; ++t) acc += gd[(int64_t)n * cnt + t] * xd[(int64_t)k * cnt + t];
        out[((int64_t)e * N + n) * K + k] = acc;
      }
    free(gd);
    free(xd);
  }
  free(P);
}

double orc_grouped_wgrad_element(const uint8_t *gq, const uint8_t *gs, const uint8_t *xq,
                                 const uint8_t *xs, const int32_t *off, int E, int64_t Mcap,
                                 int e, int n, int k) {
  int64_t *P = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
  orc_padded_starts(off, E, P);
  const int cnt = off[e + 1] - off[e];
  double acc = 0.0;
  for (int t = 0; t < cnt; ++t)
    acc += deq(gq, gs, Mcap, n, P[e] + t) * deq(xq, xs, Mcap, k, P[e] + t);
  free(P);
  return acc;
}

/* ------------------------------------------------------------------- dgrad */

/* The dgrad page's expert_for_row: start at expert 0 and step forward while a
 * next expert exists and the row is at or past that expert's first row. */
int orc_expert_for_row_scan(const int32_t *off, int E, int row) {
  int e = 0;
  while (e + 1 < E && row >= off[e + 1]) ++e;
  return e;
}

int orc_expert_for_row_bsearch(const int32_t *off, int E, int row) {
  /* largest e in [0, E) with off[e] <= row */
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (off[mid] <= row)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

/* The dgrad page's per-element path (the one it takes for tiles that straddle
 * experts): dx[row, k] = sum over n of dy[row, n] * W[e(row), n, k], with W
 * laid out [E, out_features, in_features].  Summed here in fp64. */
double orc_grouped_dgrad_element(const float *dy, const float *W, const int32_t *off, int E,
                                 int rows, int out_f, int in_f, int r, int k, double *bound_out) {
  (void)rows;
  const int e = orc_expert_for_row_scan(off, E, r);
  double acc = 0.0, bnd = 0.0;
  for (int n = 0; n < out_f; ++n) {
    const double a = (double)dy[(int64_t)r * out_f + n];
    const double w = (double)W[((int64_t)e * out_f + n) * in_f + k];
    acc += a * w;
    bnd += fabs(a) * fabs(w);
  }
  if (bound_out) *bound_out = bnd;
  return acc;
}

void orc_grouped_dgrad(const float *dy, const float *W, const int32_t *off, int E, int rows,
                       int out_f, int in_f, double *dx, double *bound) {
  for (int r = 0; r < rows; ++r)
    for (int k = 0; k < in_f; ++k) {
      double b = 0.0;
      dx[(int64_t)r * in_f + k] =
          orc_grouped_dgrad_element(dy, W, off, E, rows, out_f, in_f, r, k, &b);
      if (bound) bound[(int64_t)r * in_f + k] = b;
    }
}

/* The dgrad page's own fp32 formulation, restated as a cross-check of the fp64
 * definition above (it is not the definition).  Rows are taken in groups of 32.  A
 * group whose first and last rows map to the same expert multiplies all its rows by that
 * expert's weights; a group that straddles an expert boundary looks up each row's expert
 * on its own.  Each output is a running fp32 sum over the output features in order; the
 * page's shared-memory tiling of n and k does not change that order.  The page leaves
 * open whether a product is fused into the sum, so both readings are offered:
 * fused != 0 takes fmaf, fused == 0 rounds the product first. */
void orc_grouped_dgrad_page_f32(const float *dy, const float *W, const int32_t *off, int E,
                                int rows, int out_f, int in_f, int fused, float *dx) {
  for (int base = 0; base < rows; base += 32) {
    const int end = base + 32 < rows ? base + 32 : rows;
    const int e_first = orc_expert_for_row_scan(off, E, base);
    const int e_last = orc_expert_for_row_scan(off, E, end - 1);
    for (int r = base; r < end; ++r) {
      const int e = e_first == e_last ? e_first : orc_expert_for_row_scan(off, E, r);
      const float *a = dy + (int64_t)r * out_f;
      const float *w = W + (int64_t)e * out_f * in_f;
      for (int k = 0; k < in_f; ++k) {
        float sum = 0.0f;
        for (int n = 0; n < out_f; ++n) {
          const float wv = w[(int64_t)n * in_f + k];
          if (fused) {
            sum = fmaf(a[n], wv, sum);
          } else {
            const float prod = a[n] * wv;
            sum = sum + prod;
          }
        }
        dx[(int64_t)r * in_f + k] = sum;
      }
    }
  }
}

/* ------------------------------------------- forward and data-gradient GEMMs */

/* The post-attn page stages every routed token's activations for its expert GEMMs as
 * MXFP8 along the hidden axis: one e8m0 byte per 32 consecutive hidden features of a
 * token (its XSC_WORDS = HIDDEN / 32 scale words per token row, and mx8_scale / mx8_q
 * applied per 32-block).  Same rules as orc_mxfp8_quantize, blocks along a row. */
void orc_mxfp8_quantize_rows(const uint16_t *src, int M, int C, const int32_t *off, int E,
                             int64_t Mcap, int rule, uint8_t *q, uint8_t *sc) {
  (void)M;
  const int nb = C / 32;
  memset(q, 0, (size_t)Mcap * (size_t)C);
  memset(sc, 0, (size_t)Mcap * (size_t)nb);
  int64_t *P = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
  orc_padded_starts(off, E, P);
  for (int e = 0; e < E; ++e) {
    const int cnt = off[e + 1] - off[e];
    for (int i = 0; i < cnt; ++i) {
      const uint16_t *row = src + (int64_t)(off[e] + i) * C;
      const int64_t p = P[e] + i;
      for (int j = 0; j < nb; ++j) {
        double amax = 0.0;
        for (int c = 32 * j; c < 32 * j + 32; ++c) {
          const double v = fabs(orc_bf16_decode(row[c]));
          if (v > amax) amax = v;
        }
        const uint8_t byte = rule ? orc_mx_scale_byte_ceil448(amax) : orc_mx_scale_byte(amax);
        const int s = (int)byte - 127;
        sc[p * nb + j] = byte;
        for (int c = 32 * j; c < 32 * j + 32; ++c)
          q[p * C + c] = orc_e4m3_encode_rne_satfinite(ldexp(orc_bf16_decode(row[c]), -s));
      }
    }
  }
  free(P);
}

/* Dot product of two MXFP8 vectors of L elements (L a multiple of 32), each with one
 * e8m0 scale per 32 consecutive elements: sum_l deq(a)[l] * deq(b)[l] in fp64.  Every
 * product is exact in fp64; only the sum rounds. */
double orc_mx_dot(const uint8_t *aq, const uint8_t *as, const uint8_t *bq, const uint8_t *bs,
                  int L) {
  double acc = 0.0;
  for (int l = 0; l < L; ++l)
    acc += orc_e4m3_decode(aq[l]) * orc_e8m0_decode(as[l / 32]) *
           (orc_e4m3_decode(bq[l]) * orc_e8m0_decode(bs[l / 32]));
  return acc;
}

/* Expert of routed row r: the one whose row range [off[e], off[e+1]) holds it (the
 * dgrad page's expert_for_row; empty experts hold no rows). */
static int expert_of(const int32_t *off, int E, int r) {
  return orc_expert_for_row_bsearch(off, E, r);
}

/* The post-attn page's expert GEMMs in the forward direction: each routed token's row
 * times the transpose of its expert's weight matrix (W[e] stored [N, K], output features
 * by hidden), both operands MXFP8 along the hidden axis K. */
void orc_grouped_fprop_mx(const uint8_t *xq, const uint8_t *xs, const uint8_t *wq,
                          const uint8_t *ws, const int32_t *off, const int32_t *w_off, int E,
                          int M, int N, int K, int64_t Mcap, double *out) {
  (void)Mcap;
  const int nb = K / 32;
  int64_t *P = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
  int64_t *Pw = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
  orc_padded_starts(off, E, P);
  orc_padded_starts(w_off, E, Pw);
  for (int r = 0; r < M; ++r) {
    const int e = expert_of(off, E, r);
    const int64_t p = P[e] + (r - off[e]);
    for (int n = 0; n < N; ++n) {
      const int64_t wr = Pw[e] + n; /* row of W[e][n] */
      out[(int64_t)r * N + n] =
          orc_mx_dot(xq + p * K, xs + p * nb, wq + wr * K, ws + wr * nb, K);
    }
  }
  free(P);
  free(Pw);
}

/* The dgrad page's dx[row, k] = sum_n dy[row, n] * W[e(row), n, k] with both operands in
 * MXFP8 along n (the contraction axis): dy row-wise, W per expert along its n axis. */
void orc_grouped_dgrad_mx(const uint8_t *dyq, const uint8_t *dys, const uint8_t *wtq,
                          const uint8_t *wts, const int32_t *off, const int32_t *w_off, int E,
                          int M, int N, int K, int64_t Mcap, int64_t Mw, double *out) {
  (void)Mcap;
  const int nb = N / 32;
  int64_t *P = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
  int64_t *Pw = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E + 1));
  orc_padded_starts(off, E, P);
  orc_padded_starts(w_off, E, Pw);
  for (int r = 0; r < M; ++r) {
    const int e = expert_of(off, E, r);
    const int64_t p = P[e] + (r - off[e]);
    for (int k = 0; k < K; ++k) {
      /* W[e][n][k] for n = 0.. is row k of wtq from column Pw[e] (a multiple of 128) */
      const uint8_t *wrow = wtq + (int64_t)k * Mw + Pw[e];
      const uint8_t *wsc = wts + (int64_t)k * (Mw / 32) + Pw[e] / 32;
      out[(int64_t)r * K + k] = orc_mx_dot(dyq + p * N, dys + p * nb, wrow, wsc, N);
    }
  }
  free(P);
  free(Pw);
}
