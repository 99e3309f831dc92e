// Device arithmetic of the FP8 block quantiser, shared by every kernel that
// quantises (so that they produce identical bytes): exact scale exponent,
// power-of-two reciprocal, E4M3 packing, bf16 unpacking.
// DeepGEMM FP8 article (nxmr.cn), "补偿机制一" and "FP8 的精度陷阱".
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace bsf {

// Least e with amax <= 448 * 2**e for a finite, non-negative float amax
// (0 for amax == 0), clamped to [-126, 127].  With amax = 1.f * 2**(E-127)
// and 448 = 1.75 * 2**8: e = E - 135, plus one when the fraction f > 0.75
// (mantissa bits > 0x600000).  fp32 subnormals lie far below 448 * 2**-126.
__device__ __forceinline__ int block_exponent(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  if (bits == 0) return 0;
  const int ef = static_cast<int>(bits >> 23);
  if (ef == 0) return -126;
  int e = ef - 135 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -126 ? -126 : (e > 127 ? 127 : e);
}

// 2**-e as a float for e in [-126, 126].
__device__ __forceinline__ float inv_pow2(int e) {
  const int be = 127 - (e > 126 ? 126 : e);
  return __uint_as_float(static_cast<uint32_t>(be) << 23);
}

__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

}  // namespace bsf

// ---------------------------------------------------------------------------
// NVFP4 ("AsymGEMM" README, "FP4 Asymmetric GEMM": E2M1 data, E4M3 scales;
// "CuTeDSL bei Perplexity": one scale per 16 elements).

namespace bsf {

// 2**j as a float for j in [-126, 127] (exact).
__device__ __forceinline__ float pow2f(int j) { return __uint_as_float(static_cast<uint32_t>(127 + j) << 23); }

// E4M3 code of a non-negative float: nearest, ties to even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_code(float s) {
  const __nv_fp8x2_storage_t v = __nv_cvt_float2_to_fp8x2(make_float2(s, 0.f), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(v) & 0xFFu;
}

// Value of a non-negative E4M3 code (0x00..0x7E), exact: exponent field 0 is
// the subnormal m * 2**-9, otherwise (1 + m/8) * 2**(e - 7).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  if (e == 0) return static_cast<float>(m) * 0.001953125f;
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Eight floats -> eight E2M1 codes in one word (nearest, ties to even,
// saturating at 6); element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t pack8_e2m1(const float (&v)[8]) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return out;
}

// One block of 16 values with tensor exponent j: returns the scale code and
// writes the 16 element codes as two words.  scale = E4M3(amax / 6 * 2**-j),
// element = E2M1(x / (scale * 2**j)), each step one float32 operation rounded
// to nearest; a zero scale stores zero codes.
__device__ __forceinline__ uint32_t nvfp4_block(const float (&x)[16], int j, uint32_t& lo, uint32_t& hi) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float s = __fmul_rn(__fdiv_rn(amax, 6.0f), pow2f(-j));
  const uint32_t code = e4m3_code(s);
  const float den = e4m3_value(code) * pow2f(j);      // exact
  float y[8];
  if (code == 0) {
    lo = hi = 0u;
    return 0u;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(x[i], den);
  lo = pack8_e2m1(y);
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(x[8 + i], den);
  hi = pack8_e2m1(y);
  return code;
}

}  // namespace bsf
