// Quantisers: bf16 -> FP8 E4M3 with power-of-two (UE8M0) block scales, the
// weight scale-factor transform, and the tiled weight layout.
//
// DeepGEMM FP8 article (nxmr.cn), "补偿机制一": every scale is an exact power
// of two, packed as UE8M0 bytes four to an int32; "补偿机制三": SFs are
// MN-major with a 16-byte aligned stride; weight SFs are transformed once.
// "FP8 的精度陷阱": E4M3 = 1/4/3 bits, range +-448.
#include "common.cuh"
#include "host_utils.h"
#include "quant_math.cuh"

namespace bsf {
namespace {

// One warp per (row, group of four 128-wide K-blocks): lane l covers
// elements 16 l .. 16 l + 15 of the 512-wide group, i.e. block l / 8.
// With row_token (a packed operand's token_of_row) only rows t < *rows_used with row_token[t] >= 0
// are quantised; the others are left unwritten.
__global__ void __launch_bounds__(256) quantise_act_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t K,
                                                           uint8_t* __restrict__ q, int32_t* __restrict__ sf,
                                                           int64_t sf_ld, const int32_t* __restrict__ row_token,
                                                           const int32_t* __restrict__ rows_used) {
  pdl_launch_dependents();     // a dependent GEMM may be scheduled now; it waits for completion
  const int64_t n_groups = (K + 511) / 512;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= T * n_groups) return;
  const int64_t t = gw / n_groups;
  const int64_t g = gw - t * n_groups;
  if (row_token != nullptr && (t >= __ldg(rows_used) || __ldg(row_token + t) < 0)) return;   // whole warp
  const int64_t k0 = g * 512 + lane * 16;
  const bool active = k0 < K;

  float v[16];
  float amax = 0.f;
  if (active) {
    const uint4* src = reinterpret_cast<const uint4*>(x + t * K + k0);
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    float fa[8], fb[8];
    bf16x8_to_float(a, fa);
    bf16x8_to_float(b, fb);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = fa[i];
      v[8 + i] = fb[i];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  // max over the 8 lanes of this K-block
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  const int e = block_exponent(amax);
  if (active) {
    const float s = inv_pow2(e);
    uint4 out;
    out.x = pack4_e4m3(v[0] * s, v[1] * s, v[2] * s, v[3] * s);
    out.y = pack4_e4m3(v[4] * s, v[5] * s, v[6] * s, v[7] * s);
    out.z = pack4_e4m3(v[8] * s, v[9] * s, v[10] * s, v[11] * s);
    out.w = pack4_e4m3(v[12] * s, v[13] * s, v[14] * s, v[15] * s);
    *reinterpret_cast<uint4*>(q + t * K + k0) = out;
  }
  // byte j of the SF word = block j of the group (127 for blocks past K)
  uint32_t byte = active ? static_cast<uint32_t>(e + 127) : 127u;
  const uint32_t b0 = __shfl_sync(0xffffffffu, byte, 0);
  const uint32_t b1 = __shfl_sync(0xffffffffu, byte, 8);
  const uint32_t b2 = __shfl_sync(0xffffffffu, byte, 16);
  const uint32_t b3 = __shfl_sync(0xffffffffu, byte, 24);
  if (lane == 0) sf[g * sf_ld + t] = static_cast<int32_t>(b0 | (b1 << 8) | (b2 << 16) | (b3 << 24));
}

// One CTA (256 threads) per 128 x 128 weight block.
__global__ void __launch_bounds__(256) quantise_weight_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                              uint8_t* __restrict__ q, float* __restrict__ sf128) {
  const int64_t nkb = K / 128, nnb = N / 128;
  const int64_t blk = blockIdx.x;
  const int64_t e = blk / (nnb * nkb);
  const int64_t rem = blk - e * nnb * nkb;
  const int64_t nb = rem / nkb, kb = rem - nb * nkb;
  // thread -> (row r in 0..127 step 16 per pass, 16-element column chunk c in 0..7)
  const int c = threadIdx.x & 7;
  const int r0 = threadIdx.x >> 3;  // 0..31
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
  const int ex = block_exponent(amax);
  const float s = inv_pow2(ex);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int64_t row = nb * 128 + r0 + 32 * p;
    uint4 out;
    out.x = pack4_e4m3(v[p][0] * s, v[p][1] * s, v[p][2] * s, v[p][3] * s);
    out.y = pack4_e4m3(v[p][4] * s, v[p][5] * s, v[p][6] * s, v[p][7] * s);
    out.z = pack4_e4m3(v[p][8] * s, v[p][9] * s, v[p][10] * s, v[p][11] * s);
    out.w = pack4_e4m3(v[p][12] * s, v[p][13] * s, v[p][14] * s, v[p][15] * s);
    *reinterpret_cast<uint4*>(q + (e * N + row) * K + kb * 128 + c * 16) = out;
  }
  if (threadIdx.x == 0) sf128[(e * nnb + nb) * nkb + kb] = __uint_as_float(static_cast<uint32_t>(ex + 127) << 23);
}

// One thread per output word [e][i][n].
__global__ void prepare_weight_sf_kernel(const float* __restrict__ sf128, int64_t E, int64_t N, int64_t K,
                                         int32_t* __restrict__ sfb, int* err) {
  const int64_t nkb = K / 128, nnb = N / 128, nw = (nkb + 3) / 4;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= E * nw * N) return;
  const int64_t n = idx % N;
  const int64_t i = (idx / N) % nw;
  const int64_t e = idx / (N * nw);
  uint32_t word = 0;
  int bad = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t kb = 4 * i + j;
    uint32_t byte = 127;
    if (kb < nkb) {
      const uint32_t bits = __float_as_uint(sf128[(e * nnb + n / 128) * nkb + kb]);
      const uint32_t be = bits >> 23;
      if ((bits & 0x807FFFFFu) != 0 || be == 0 || be == 255) {
        bad = 1;                      // not a positive, normal power of two
      } else {
        byte = be;                    // UE8M0 byte = biased float32 exponent
      }
    }
    word |= byte << (8 * j);
  }
  if (bad) raise_error(err, BSF_DEVERR_BAD_SCALE);
  sfb[idx] = static_cast<int32_t>(word);
}

// Weight tiling: one thread per 16 output bytes.  Output block (e, nt, kb) is
// the 128 x 128-byte piece of expert e at rows 128 nt.., bytes 128 kb.., its
// rows 128 bytes apart; eight consecutive threads read one 128-byte row piece.
__global__ void __launch_bounds__(256) tile_weights_kernel(const uint4* __restrict__ b, int64_t N, int64_t row_bytes,
                                                           int64_t n16, uint4* __restrict__ out) {
  const int64_t nkb = row_bytes / 128, nnt = N / 128, row16 = row_bytes / 16;
  for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < n16;
       o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t blk = o / 1024, r = (o / 8) % 128, c16 = o % 8;
    const int64_t kb = blk % nkb, nt = (blk / nkb) % nnt, e = blk / (nkb * nnt);
    out[o] = __ldg(b + (e * N + nt * 128 + r) * row16 + kb * 8 + c16);
  }
}

}  // namespace
}  // namespace bsf

using namespace bsf;

extern "C" bsf_status bsf_tile_weights(const uint8_t* b, int64_t E, int64_t N, int64_t row_bytes, uint8_t* out,
                                       bsf_stream_t stream) {
  if (E <= 0 || N <= 0 || row_bytes <= 0 || N % 128 || row_bytes % 128) return BSF_ERR_INVALID_ARGUMENT;
  if (!b || !out || b == out) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(b) || !aligned16(out)) return BSF_ERR_MISALIGNED;
  if (!fits_weights(E, N, row_bytes)) return BSF_ERR_UNSUPPORTED;
  if (E * N > INT32_MAX || E * N * (row_bytes / 128) > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  const int64_t n16 = E * N * row_bytes / 16;
  int64_t blocks = static_cast<int64_t>(sm_count()) * 8;
  const int64_t need = (n16 + 255) / 256;
  if (need < blocks) blocks = need;
  tile_weights_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(b), N, row_bytes, n16, reinterpret_cast<uint4*>(out));
  return launch_status();
}

extern "C" bsf_status bsf_quantise_act(const void* x, int64_t T, int64_t K, uint8_t* q, int32_t* sf, int64_t sf_ld,
                                       bsf_stream_t stream) {
  if (T < 0 || K <= 0 || K % 128 != 0) return BSF_ERR_INVALID_ARGUMENT;
  if (T == 0) return BSF_OK;
  if (!x || !q || !sf) return BSF_ERR_INVALID_ARGUMENT;
  if (sf_ld < T || sf_ld % 4 != 0) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return BSF_ERR_MISALIGNED;
  if (!fits_rows(T, K)) return BSF_ERR_UNSUPPORTED;
  const int64_t warps = T * ((K + 511) / 512);
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  quantise_act_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(x), T, K, q, sf, sf_ld, nullptr, nullptr);
  return launch_status();
}

extern "C" bsf_status bsf_quantise_act_rows(const void* x, int64_t T, int64_t K, const int32_t* token_of_row,
                                            const int32_t* rows_used, uint8_t* q, int32_t* sf, int64_t sf_ld,
                                            bsf_stream_t stream) {
  if (T < 0 || K <= 0 || K % 128 != 0) return BSF_ERR_INVALID_ARGUMENT;
  if (T == 0) return BSF_OK;
  if (!x || !q || !sf || !token_of_row || !rows_used) return BSF_ERR_INVALID_ARGUMENT;
  if (sf_ld < T || sf_ld % 4 != 0) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return BSF_ERR_MISALIGNED;
  if (!fits_rows(T, K)) return BSF_ERR_UNSUPPORTED;
  const int64_t warps = T * ((K + 511) / 512);
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  quantise_act_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(x), T, K, q, sf, sf_ld, token_of_row, rows_used);
  return launch_status();
}

extern "C" bsf_status bsf_quantise_weight(const void* w, int64_t E, int64_t N, int64_t K, uint8_t* q, float* sf128,
                                          bsf_stream_t stream) {
  if (E < 0 || N <= 0 || K <= 0 || N % 128 || K % 128) return BSF_ERR_INVALID_ARGUMENT;
  if (E == 0) return BSF_OK;
  if (!w || !q || !sf128) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(w) || !aligned16(q)) return BSF_ERR_MISALIGNED;
  if (!fits_weights(E, N, K)) return BSF_ERR_UNSUPPORTED;
  const int64_t blocks = E * (N / 128) * (K / 128);
  if (blocks > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  quantise_weight_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(w), N, K, q, sf128);
  return launch_status();
}

extern "C" bsf_status bsf_prepare_weight_sf(const float* sf128, int64_t E, int64_t N, int64_t K, int32_t* sfb,
                                            bsf_stream_t stream) {
  if (E < 0 || N <= 0 || K <= 0 || N % 128 || K % 128) return BSF_ERR_INVALID_ARGUMENT;
  if (E == 0) return BSF_OK;
  if (!sf128 || !sfb) return BSF_ERR_INVALID_ARGUMENT;
  if (!fits_weights(E, N, K)) return BSF_ERR_UNSUPPORTED;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  const int64_t total = E * ((K / 128 + 3) / 4) * N;
  const int64_t blocks = (total + 255) / 256;
  if (blocks > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  prepare_weight_sf_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      sf128, E, N, K, sfb, err);
  return launch_status();
}
