// Weighted combine (un-permute) of the expert outputs.
//
// "GEMM 执行方式" §4.4 / §4.6: z_t = sum_r p[t, r] * y_packed[output_index[t, r]]
// (ep_gather reads only valid rows).  "CuTeDSL bei Perplexity": the combine
// kernel accumulates in registers with vectorised loads, using the offsets
// computed at dispatch.
//
// One warp per (token, 256-column slice): each lane owns 8 consecutive bf16
// columns (one 16-byte load per route), accumulates in FP32 in r order and
// stores 16 bytes of bf16 (round to nearest even).
#include "common.cuh"
#include "host_utils.h"

namespace bsf {
namespace {

constexpr int kMaxKr = 32;

// At most 64 registers (four CTAs per SM): with 66 the kernel held three and large batches ran
// 11-12 % slower (bandwidth-bound, occupancy-limited; same-box A/B, bit-identical output).
__global__ void __launch_bounds__(256, 4) combine_kernel(const uint16_t* __restrict__ y, int64_t y_rows,
                                                      const int32_t* __restrict__ output_index,
                                                      const float* __restrict__ topk_weights, int64_t T, int kr,
                                                      int64_t N, uint16_t* __restrict__ z) {
  const int64_t slices = (N + 255) / 256;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= T * slices) return;
  const int64_t t = gw / slices;
  const int64_t col = (gw - t * slices) * 256 + lane * 8;
  // route r's row and weight live in lane r (kr <= 32)
  int my_row = -1;
  float my_p = 0.f;
  if (lane < kr) {
    my_row = output_index[t * kr + lane];
    my_p = topk_weights[t * kr + lane];
    if (my_row >= y_rows) my_row = -1;
  }
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const bool active = col < N;
  // routes in groups of 8: all loads of a group are issued before any is used
  for (int r0 = 0; r0 < kr; r0 += 8) {
    uint4 v[8];
    float pr[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, (r0 + j) & 31);
      pr[j] = __shfl_sync(0xffffffffu, my_p, (r0 + j) & 31);
      const bool use = active && r0 + j < kr && row >= 0;
      v[j] = use ? __ldg(reinterpret_cast<const uint4*>(y + static_cast<int64_t>(row) * N + col))
                 : make_uint4(0, 0, 0, 0);
      if (!use) pr[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (r0 + j >= kr) break;
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(pr[j], __uint_as_float(w[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(pr[j], __uint_as_float(w[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
  }
  if (!active) return;
  uint4 out;
  out.x = pack_bf16x2(acc[0], acc[1]);
  out.y = pack_bf16x2(acc[2], acc[3]);
  out.z = pack_bf16x2(acc[4], acc[5]);
  out.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(z + t * N + col) = out;
}

}  // namespace
}  // namespace bsf

using namespace bsf;

extern "C" bsf_status bsf_combine(const void* y, int64_t y_rows, const int32_t* output_index,
                                  const float* topk_weights, int64_t T, int64_t kr, int64_t N, void* z,
                                  bsf_stream_t stream) {
  if (T < 0 || kr <= 0 || kr > kMaxKr || N <= 0 || N % 8 || y_rows < 0) return BSF_ERR_INVALID_ARGUMENT;
  if (T == 0) return BSF_OK;
  if (!y || !output_index || !topk_weights || !z) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(y) || !aligned16(z)) return BSF_ERR_MISALIGNED;
  if (!fits_rows(T, N)) return BSF_ERR_UNSUPPORTED;
  const int64_t warps = T * ((N + 255) / 256);
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  combine_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(y), y_rows, output_index, topk_weights, T, static_cast<int>(kr), N,
      static_cast<uint16_t*>(z));
  return launch_status();
}
