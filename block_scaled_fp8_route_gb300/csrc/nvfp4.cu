// NVFP4 quantisers and the per-tensor (per-expert) exponent.
//
// "AsymGEMM" README, "FP4 Asymmetric GEMM": FP4 data is E2M1 packed two
// elements per byte with FP8 E4M3 scale factors.  "CuTeDSL bei Perplexity"
// (Blackwell support): the NVFP4 quantiser takes the absolute maximum over 16
// elements.  A power-of-two tensor scale 2**j widens the range of the E4M3
// block scales (a block's scale is E4M3(amax / 6 / 2**j)); the grouped GEMM
// multiplies its FP32 accumulator by 2**(j_A + j_B) exactly.
//
// Layouts: data row-major, 2 elements per byte (element 2i in the low nibble
// of byte i); scales as int32 words of four UE4M3 bytes, byte i for elements
// 64w + 16i .. 64w + 16i + 15 of word w, MN-major.
#include "common.cuh"
#include "host_utils.h"
#include "quant_math.cuh"

namespace bsf {
namespace {

constexpr int kJLimit = 100;

__device__ __forceinline__ int clamp_j(int j) { return j < -kJLimit ? -kJLimit : (j > kJLimit ? kJLimit : j); }

// One thread per (row, 64-element word w), rows fastest so that the scale
// words of a warp are 32 consecutive int32.  Row r belongs to group
// r / group_rows (an expert for weights, the whole tensor for activations);
// its scale word lives at ((group * nwords) + w) * ld + r % group_rows.
__global__ void __launch_bounds__(256) quantise_nvfp4_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t K,
                                                             int64_t group_rows, int j_const,
                                                             const int32_t* __restrict__ j_group,
                                                             uint8_t* __restrict__ q, int32_t* __restrict__ sf,
                                                             int64_t ld) {
  pdl_launch_dependents();     // a dependent GEMM may be scheduled now; it waits for completion
  const int64_t nwords = K / 64;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= R * nwords) return;
  const int64_t row = idx % R, w = idx / R;
  const int64_t g = row / group_rows;
  const int j = clamp_j(j_group ? j_group[g] : j_const);
  const uint4* src = reinterpret_cast<const uint4*>(x + row * K + w * 64);
  uint32_t codes[8];
  uint32_t word = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float fa[8], fb[8], f[16];
    bf16x8_to_float(__ldg(src + 2 * b), fa);
    bf16x8_to_float(__ldg(src + 2 * b + 1), fb);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[i] = fa[i];
      f[8 + i] = fb[i];
    }
    word |= nvfp4_block(f, j, codes[2 * b], codes[2 * b + 1]) << (8 * b);
  }
  uint4* dst = reinterpret_cast<uint4*>(q + row * (K / 2) + w * 32);
  dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
  sf[(g * nwords + w) * ld + row % group_rows] = static_cast<int32_t>(word);
}

// Per-group absolute maximum as float bits (non-negative floats order like
// their bit patterns).  grid = (blocks per group, groups).
__global__ void __launch_bounds__(256) group_amax_kernel(const uint16_t* __restrict__ x, int64_t per_group,
                                                         uint32_t* __restrict__ amax_bits) {
  const int64_t g = blockIdx.y;
  const uint4* src = reinterpret_cast<const uint4*>(x + g * per_group);
  const int64_t n16 = per_group / 8;
  uint32_t m = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = (w[k] << 16) & 0x7FFFFFFFu, hi = w[k] & 0x7FFF0000u;
      m = max(m, max(lo, hi));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0 && m) atomicMax(amax_bits + g, m);
}

// amax bits -> least j with amax <= 6 * 448 * 2**j (0 for amax == 0), in
// [-100, 100].  amax = (1 + f) * 2**(E - 127); 2688 = 1.3125 * 2**11, so
// j = E - 138, plus one when f > 0.3125 (mantissa bits > 0x280000).
__global__ void group_exponent_kernel(int32_t* __restrict__ inout, int64_t groups) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  const uint32_t b = static_cast<uint32_t>(inout[g]);
  int j = 0;
  if (b != 0) {
    const int ef = static_cast<int>(b >> 23);
    j = ef == 0 ? -kJLimit : ef - 138 + ((b & 0x7FFFFFu) > 0x280000u ? 1 : 0);
  }
  inout[g] = clamp_j(j);
}

bsf_status launch_quantise(const void* x, int64_t R, int64_t K, int64_t group_rows, int j_const,
                           const int32_t* j_group, uint8_t* q, int32_t* sf, int64_t ld, cudaStream_t s) {
  const int64_t threads = R * (K / 64);
  if (threads == 0) return BSF_OK;
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  quantise_nvfp4_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const uint16_t*>(x), R, K,
                                                                      group_rows, j_const, j_group, q, sf, ld);
  return launch_status();
}

}  // namespace
}  // namespace bsf

using namespace bsf;

extern "C" bsf_status bsf_quantise_act_nvfp4(const void* x, int64_t T, int64_t K, int a_exp, uint8_t* q,
                                             int32_t* sf, int64_t sf_ld, bsf_stream_t stream) {
  if (T < 0 || K <= 0 || K % 64 || a_exp < -kJLimit || a_exp > kJLimit) return BSF_ERR_INVALID_ARGUMENT;
  if (sf_ld < T || sf_ld % 4) return BSF_ERR_INVALID_ARGUMENT;
  if (T == 0) return BSF_OK;
  if (!x || !q || !sf) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return BSF_ERR_MISALIGNED;
  if (!fits_rows(T, K)) return BSF_ERR_UNSUPPORTED;
  return launch_quantise(x, T, K, T, a_exp, nullptr, q, sf, sf_ld, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" bsf_status bsf_quantise_weight_nvfp4(const void* w, int64_t E, int64_t N, int64_t K,
                                                const int32_t* b_exp, uint8_t* q, int32_t* sfb,
                                                bsf_stream_t stream) {
  if (E <= 0 || N <= 0 || K <= 0 || K % 64) return BSF_ERR_INVALID_ARGUMENT;
  if (!w || !b_exp || !q || !sfb) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(w) || !aligned16(q) || !aligned16(sfb)) return BSF_ERR_MISALIGNED;
  if (!fits_weights(E, N, K)) return BSF_ERR_UNSUPPORTED;
  return launch_quantise(w, E * N, K, N, 0, b_exp, q, sfb, N, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" bsf_status bsf_nvfp4_tensor_exponent(const void* x, int64_t groups, int64_t per_group, int32_t* exp_out,
                                                bsf_stream_t stream) {
  if (groups <= 0 || per_group <= 0 || per_group % 8) return BSF_ERR_INVALID_ARGUMENT;
  if (!x || !exp_out) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(x)) return BSF_ERR_MISALIGNED;
  if (groups > 65535) return BSF_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(exp_out, 0, static_cast<size_t>(groups) * sizeof(int32_t), s) != cudaSuccess)
    return BSF_ERR_CUDA;
  int64_t per_block = 256 * 8 * 16;                       // 16 uint4 per thread
  int64_t bx = (per_group + per_block - 1) / per_block;
  const int64_t cap = (4 * static_cast<int64_t>(sm_count()) + groups - 1) / groups;
  if (bx > cap) bx = cap;
  if (bx < 1) bx = 1;
  group_amax_kernel<<<dim3(static_cast<unsigned>(bx), static_cast<unsigned>(groups)), 256, 0, s>>>(
      static_cast<const uint16_t*>(x), per_group, reinterpret_cast<uint32_t*>(exp_out));
  group_exponent_kernel<<<static_cast<unsigned>((groups + 255) / 256), 256, 0, s>>>(exp_out, groups);
  return launch_status();
}
