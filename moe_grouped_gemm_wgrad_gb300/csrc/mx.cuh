// MXFP8 element and scale arithmetic shared by the quantizers: the e8m0 scale byte of a
// 32-element block from its largest magnitude, and the saturating round-to-nearest-even
// e4m3 convert.
#pragma once
#include <cuda_fp8.h>

#include <cstdint>

namespace mgw {

__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// Rule 0 (OCP MX): floor(log2 amax) is the bf16 exponent field minus 127 for normal
// values; the scale byte is that minus 8 plus the bias 127, clamped at 0 (which also
// covers amax == 0 and every subnormal amax).
// Rule 1 (the post-attn page's RoundUp): the biased exponent of amax * fp32(1/448)
// rounded up to a power of two, clamped to [1, 254].
// Returns the byte; *inv = 2^(127 - byte) (exact; subnormal for byte 254).
__device__ __forceinline__ int scale_byte(uint32_t amax_bits, int rule, float* inv) {
  int byte;
  if (rule == 0) {
    const int ef = static_cast<int>(amax_bits >> 7);
    byte = ef > 8 ? ef - 8 : 0;
  } else {
    const float r = __fmul_rn(__uint_as_float(amax_bits << 16), 1.0f / 448.0f);
    const uint32_t rb = __float_as_uint(r);
    byte = static_cast<int>((rb >> 23) & 0xFFu) + ((rb & 0x7FFFFFu) != 0u ? 1 : 0);
    byte = min(max(byte, 1), 254);
  }
  *inv = byte < 254 ? __uint_as_float(static_cast<uint32_t>(254 - byte) << 23)
                    : __uint_as_float(0x00400000u);
  return byte;
}

}  // namespace mgw
