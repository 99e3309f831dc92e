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
