// FP8 E4M3 quantisers with float32 scale factors (the scales are not cast to UE8M0).
//
// "AsymGEMM" README, notation: disable_ue8m0_cast keeps the scale factors in
// float32.  DeepGEMM article, "补偿机制一": a float32 scale that is not a power
// of two is applied with rounding.  Per block (1 x 128 for activations,
// 128 x 128 for weights): s = amax / 448 (one float32 division, nearest even;
// 1 for an all-zero block), q = E4M3(x / s) (one float32 division, then
// nearest-even E4M3, saturating).
#include "common.cuh"
#include "host_utils.h"
#include "quant_math.cuh"

namespace bsf {
namespace {

__device__ __forceinline__ float f32_scale(float amax) { return amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f); }

__device__ __forceinline__ uint4 quantise16_div(const float (&v)[16], float s) {
  float y[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] = __fdiv_rn(v[i], s);
  uint4 out;
  out.x = pack4_e4m3(y[0], y[1], y[2], y[3]);
  out.y = pack4_e4m3(y[4], y[5], y[6], y[7]);
  out.z = pack4_e4m3(y[8], y[9], y[10], y[11]);
  out.w = pack4_e4m3(y[12], y[13], y[14], y[15]);
  return out;
}

// One warp per (row, 512 values): lane l covers values 16 l .. 16 l + 15, block l / 8.
__global__ void __launch_bounds__(256) quantise_act_f32sf_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t K,
                                                                 uint8_t* __restrict__ q, float* __restrict__ sf,
                                                                 int64_t sf_ld) {
  pdl_launch_dependents();
  const int64_t n_groups = (K + 511) / 512;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= T * n_groups) return;
  const int64_t t = gw / n_groups, g = gw - t * n_groups;
  const int64_t k0 = g * 512 + lane * 16;
  const bool active = k0 < K;
  float v[16];
  float amax = 0.f;
  if (active) {
    const uint4* src = reinterpret_cast<const uint4*>(x + t * K + k0);
    float fa[8], fb[8];
    bf16x8_to_float(__ldg(src), fa);
    bf16x8_to_float(__ldg(src + 1), fb);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = fa[i];
      v[8 + i] = fb[i];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  const float s = f32_scale(amax);
  if (active) {
    *reinterpret_cast<uint4*>(q + t * K + k0) = quantise16_div(v, s);
    if ((lane & 7) == 0) sf[(k0 / 128) * sf_ld + t] = s;
  }
}

// One CTA (256 threads) per 128 x 128 weight block.
__global__ void __launch_bounds__(256) quantise_weight_f32sf_kernel(const uint16_t* __restrict__ w, int64_t N,
                                                                    int64_t K, uint8_t* __restrict__ q,
                                                                    float* __restrict__ sf) {
  const int64_t nkb = K / 128, nnb = N / 128;
  const int64_t blk = blockIdx.x;
  const int64_t e = blk / (nnb * nkb);
  const int64_t rem = blk - e * nnb * nkb;
  const int64_t nb = rem / nkb, kb = rem - nb * nkb;
  const int c = threadIdx.x & 7;       // 16-value column chunk
  const int r0 = threadIdx.x >> 3;     // rows r0 + 32 p
  float v[4][16];
  float amax = 0.f;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int64_t row = nb * 128 + r0 + 32 * p;
    const uint4* src = reinterpret_cast<const uint4*>(w + (e * N + row) * K + kb * 128 + c * 16);
    float fa[8], fb[8];
    bf16x8_to_float(__ldg(src), fa);
    bf16x8_to_float(__ldg(src + 1), fb);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[p][i] = fa[i];
      v[p][8 + i] = fb[i];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[p][i]));
  }
  __shared__ float warp_max[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_max[i]);
  const float s = f32_scale(amax);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int64_t row = nb * 128 + r0 + 32 * p;
    *reinterpret_cast<uint4*>(q + (e * N + row) * K + kb * 128 + c * 16) = quantise16_div(v[p], s);
  }
  if (threadIdx.x == 0) sf[(e * nnb + nb) * nkb + kb] = s;
}

}  // namespace
}  // namespace bsf

using namespace bsf;

extern "C" bsf_status bsf_quantise_act_f32sf(const void* x, int64_t T, int64_t K, uint8_t* q, float* sf,
                                             int64_t sf_ld, bsf_stream_t stream) {
  if (T < 0 || K <= 0 || K % 128) return BSF_ERR_INVALID_ARGUMENT;
  if (sf_ld < T || sf_ld % 4) return BSF_ERR_INVALID_ARGUMENT;
  if (T == 0) return BSF_OK;
  if (!x || !q || !sf) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return BSF_ERR_MISALIGNED;
  if (!fits_rows(T, K)) return BSF_ERR_UNSUPPORTED;
  const int64_t blocks = (T * ((K + 511) / 512) * 32 + 255) / 256;
  if (blocks > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  quantise_act_f32sf_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(x), T, K, q, sf, sf_ld);
  return launch_status();
}

extern "C" bsf_status bsf_quantise_weight_f32sf(const void* w, int64_t E, int64_t N, int64_t K, uint8_t* q,
                                                float* sf, bsf_stream_t stream) {
  if (E < 0 || N <= 0 || K <= 0 || N % 128 || K % 128) return BSF_ERR_INVALID_ARGUMENT;
  if (E == 0) return BSF_OK;
  if (!w || !q || !sf) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(w) || !aligned16(q)) return BSF_ERR_MISALIGNED;
  if (!fits_weights(E, N, K)) return BSF_ERR_UNSUPPORTED;
  const int64_t blocks = E * (N / 128) * (K / 128);
  if (blocks > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  quantise_weight_f32sf_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(w), N, K, q, sf);
  return launch_status();
}
