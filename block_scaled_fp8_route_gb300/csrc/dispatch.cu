// Single-launch dispatch for small batches (decode): quantise + route + scatter.
//
// "CuTeDSL bei Perplexity" (MoE dispatch, decode variant): with few tokens the
// routing information is small enough for one block, and one launch should do
// the routing and the copies.  Here every CTA recomputes the whole routing of
// the batch in shared memory (R <= 16384 assignments, E <= 256 experts: a few
// microseconds), so no grid-wide barrier is needed; each CTA then quantises
// its share of the routed rows straight from the bf16 activations into their
// packed rows (DeepGEMM FP8 article, "补偿机制一": 1 x 128 power-of-two UE8M0
// scales), and marks its share of the padding rows.  The bytes written are
// identical to quantise_act -> route -> scatter (same device arithmetic).
#include "common.cuh"
#include "host_utils.h"
#include "quant_math.cuh"
#include "route_block.cuh"

namespace bsf {
namespace {

constexpr int kMaxShare = 1024;   // routed assignments one CTA may own
static_assert(kSmallMaxR == BSF_DISPATCH_MAX_ASSIGNMENTS && kSmallMaxE == BSF_DISPATCH_MAX_EXPERTS,
              "single-launch limits out of sync with the header");

// FP4 = false: E4M3 rows with one UE8M0 byte per 128 values (bsf_quantise_act);
// FP4 = true: NVFP4 rows (K/2 bytes) with one UE4M3 byte per 16 values and
// tensor exponent a_exp (bsf_quantise_act_nvfp4).
template <bool FP4>
__global__ void __launch_bounds__(kSmallThreads) dispatch_small_kernel(
    const uint16_t* __restrict__ x, int64_t T, int64_t K, const int32_t* __restrict__ ids, int kr, int E, int layout,
    int64_t a_or_m, int64_t m_cap, int32_t* __restrict__ counts, int32_t* __restrict__ seg_start,
    int32_t* __restrict__ output_index, int32_t* __restrict__ token_of_row, int32_t* __restrict__ m_indices,
    uint8_t* __restrict__ a_packed, int32_t* __restrict__ sfa_packed, int64_t sfa_ld, int a_exp, int* err) {
  __shared__ RouteBlockSmem sm;
  __shared__ int share_tok[kMaxShare];
  __shared__ int share_dest[kMaxShare];
  __shared__ int n_share;
  pdl_launch_dependents();     // a dependent GEMM may be scheduled now; it waits for completion
  const int64_t R = T * kr;
  const int G = gridDim.x, b = blockIdx.x;
  if (threadIdx.x == 0) n_share = 0;
  // (route_in_block synchronises the CTA before any on_assign call)
  route_in_block(ids, R, E, layout, a_or_m, m_cap, sm, [&](int64_t i, int64_t dest) {
    if (i % G != b) return;
    output_index[i] = static_cast<int32_t>(dest);
    if (dest >= 0) {
      const int t = static_cast<int>(i / kr);
      token_of_row[dest] = t;
      const int s = atomicAdd(&n_share, 1);     // order of the list is irrelevant: each entry is independent
      share_tok[s] = t;
      share_dest[s] = static_cast<int>(dest);
    }
  });
  const int tid = threadIdx.x;
  if (b == 0) {
    if (tid < E) {
      const int M = sm.hist[tid];
      counts[tid] = layout == BSF_LAYOUT_MASKED ? (M < a_or_m ? M : static_cast<int>(a_or_m)) : M;
      seg_start[tid] = sm.seg[tid];
    }
    if (tid == 0) {
      seg_start[E] = sm.seg[E];
      if (sm.flags) raise_error(err, sm.flags);
    }
  }
  // padding marks and m_indices for this CTA's share of the used rows
  const int rows_used = sm.seg[E];
  for (int r = b + G * tid; r < rows_used; r += G * kSmallThreads) {
    int lo = 0, hi = E - 1;                      // last expert whose segment starts at or before r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sm.seg[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int M = sm.hist[lo];
    const int placed = layout == BSF_LAYOUT_MASKED ? (M < a_or_m ? M : static_cast<int>(a_or_m)) : M;
    if (r - sm.seg[lo] >= placed) token_of_row[r] = -1;
    if (m_indices) m_indices[r] = lo;
  }
  // quantise + scatter: one warp per (routed row, 512-wide K group), lane = 16 elements
  const int n_groups = static_cast<int>((K + 511) / 512);
  const int warp = tid >> 5, lane = tid & 31;
  const int items = n_share * n_groups;
  for (int it = warp; it < items; it += kSmallWarps) {
    const int s = it / n_groups, g = it - s * n_groups;
    const int64_t t = share_tok[s], dest = share_dest[s];
    const int64_t k0 = static_cast<int64_t>(g) * 512 + lane * 16;
    const bool active = k0 < K;
    float v[16];
    float amax = 0.f;
    if (active) {
      const uint4* src = reinterpret_cast<const uint4*>(x + t * K + k0);
      float fa[8], fb[8];
      bf16x8_to_float(__ldg(src), fa);
      bf16x8_to_float(__ldg(src + 1), fb);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = fa[j];
        v[8 + j] = fb[j];
      }
      if constexpr (!FP4) {
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
      }
    }
    if constexpr (FP4) {
      // lane = one 16-value block: 8 bytes of codes, one scale byte; lanes 4m..4m+3 form scale word m
      uint32_t lo = 0, hi = 0, code = 0;
      if (active) code = nvfp4_block(v, a_exp, lo, hi);
      if (active) *reinterpret_cast<uint2*>(a_packed + dest * (K / 2) + k0 / 2) = make_uint2(lo, hi);
      const uint32_t c1 = __shfl_down_sync(0xffffffffu, code, 1);
      const uint32_t c2 = __shfl_down_sync(0xffffffffu, code, 2);
      const uint32_t c3 = __shfl_down_sync(0xffffffffu, code, 3);
      if (active && (lane & 3) == 0)
        sfa_packed[(k0 / 64) * sfa_ld + dest] = static_cast<int32_t>(code | (c1 << 8) | (c2 << 16) | (c3 << 24));
      continue;
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const int e = block_exponent(amax);
    if (active) {
      const float sc = inv_pow2(e);
      uint4 out;
      out.x = pack4_e4m3(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
      out.y = pack4_e4m3(v[4] * sc, v[5] * sc, v[6] * sc, v[7] * sc);
      out.z = pack4_e4m3(v[8] * sc, v[9] * sc, v[10] * sc, v[11] * sc);
      out.w = pack4_e4m3(v[12] * sc, v[13] * sc, v[14] * sc, v[15] * sc);
      *reinterpret_cast<uint4*>(a_packed + dest * K + k0) = out;
    }
    const uint32_t byte = active ? static_cast<uint32_t>(e + 127) : 127u;
    const uint32_t b0 = __shfl_sync(0xffffffffu, byte, 0);
    const uint32_t b1 = __shfl_sync(0xffffffffu, byte, 8);
    const uint32_t b2 = __shfl_sync(0xffffffffu, byte, 16);
    const uint32_t b3 = __shfl_sync(0xffffffffu, byte, 24);
    if (lane == 0) sfa_packed[g * sfa_ld + dest] = static_cast<int32_t>(b0 | (b1 << 8) | (b2 << 16) | (b3 << 24));
  }
}

}  // namespace
}  // namespace bsf

using namespace bsf;

namespace bsf {
namespace {

template <bool FP4>
bsf_status launch_dispatch(const void* x, int64_t T, int64_t K, const int32_t* topk_ids, int64_t kr, int64_t E,
                           int layout, int64_t align_or_max_m, int32_t* counts, int32_t* seg_start,
                           int32_t* output_index, int32_t* token_of_row, int32_t* m_indices, int64_t m_cap,
                           uint8_t* a_packed, int32_t* sfa_packed, int64_t sfa_ld, int a_exp, bsf_stream_t stream) {
  if (T < 0 || kr <= 0 || E <= 0 || K <= 0 || K % (FP4 ? 64 : 128)) return BSF_ERR_INVALID_ARGUMENT;
  if (layout != BSF_LAYOUT_CONTIGUOUS && layout != BSF_LAYOUT_MASKED) return BSF_ERR_INVALID_ARGUMENT;
  if (align_or_max_m < 1 || a_exp < -100 || a_exp > 100) return BSF_ERR_INVALID_ARGUMENT;
  if (T > kSmallMaxR / kr) return BSF_ERR_UNSUPPORTED;   // before forming R, which must not wrap
  const int64_t R = T * kr;
  if (R > kSmallMaxR || E > kSmallMaxE) return BSF_ERR_UNSUPPORTED;
  if (!x || !topk_ids || !counts || !seg_start || !output_index || !token_of_row || !a_packed || !sfa_packed)
    return BSF_ERR_INVALID_ARGUMENT;
  const int64_t need_cap = layout == BSF_LAYOUT_MASKED ? E * align_or_max_m : R + E * (align_or_max_m - 1);
  if (m_cap < need_cap || m_cap > INT32_MAX) return BSF_ERR_INVALID_ARGUMENT;
  if (sfa_ld < m_cap || sfa_ld % 4) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(a_packed) || !aligned16(sfa_packed)) return BSF_ERR_MISALIGNED;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  // each CTA owns at most kMaxShare assignments; use every SM when the batch allows
  int64_t grid = sm_count();
  const int64_t min_grid = (R + kMaxShare - 1) / kMaxShare;
  if (grid < min_grid) grid = min_grid;
  if (R > 0 && grid > R) grid = R;
  if (grid < 1) grid = 1;
  dispatch_small_kernel<FP4><<<static_cast<unsigned>(grid), kSmallThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(x), T, K, topk_ids, static_cast<int>(kr), static_cast<int>(E), layout,
      align_or_max_m, m_cap, counts, seg_start, output_index, token_of_row, m_indices, a_packed, sfa_packed, sfa_ld,
      a_exp, err);
  return launch_status();
}

}  // namespace
}  // namespace bsf

extern "C" bsf_status bsf_dispatch(const void* x, int64_t T, int64_t K, const int32_t* topk_ids, int64_t kr, int64_t E,
                                   int layout, int64_t align_or_max_m, int32_t* counts, int32_t* seg_start,
                                   int32_t* output_index, int32_t* token_of_row, int32_t* m_indices, int64_t m_cap,
                                   uint8_t* a_packed, int32_t* sfa_packed, int64_t sfa_ld, bsf_stream_t stream) {
  return launch_dispatch<false>(x, T, K, topk_ids, kr, E, layout, align_or_max_m, counts, seg_start, output_index,
                                token_of_row, m_indices, m_cap, a_packed, sfa_packed, sfa_ld, 0, stream);
}

extern "C" bsf_status bsf_dispatch_nvfp4(const void* x, int64_t T, int64_t K, int a_exp, const int32_t* topk_ids,
                                         int64_t kr, int64_t E, int layout, int64_t align_or_max_m, int32_t* counts,
                                         int32_t* seg_start, int32_t* output_index, int32_t* token_of_row,
                                         int32_t* m_indices, int64_t m_cap, uint8_t* a_packed, int32_t* sfa_packed,
                                         int64_t sfa_ld, bsf_stream_t stream) {
  return launch_dispatch<true>(x, T, K, topk_ids, kr, E, layout, align_or_max_m, counts, seg_start, output_index,
                               token_of_row, m_indices, m_cap, a_packed, sfa_packed, sfa_ld, a_exp, stream);
}
