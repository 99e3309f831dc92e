// Routing of a small batch inside one CTA: histogram, segment starts and
// stable ranks (ascending flat index t * k_r + r inside each expert).
// "GEMM 执行方式" §4.2-§4.6; "CuTeDSL bei Perplexity": decode batches carry
// little routing information and are routed by a single block.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace bsf {

constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallMaxE = 256;
constexpr int64_t kSmallMaxR = 16384;

struct RouteBlockSmem {
  int hist[kSmallMaxE];                 // M_e
  int base[kSmallMaxE];                 // running rank base per expert
  int seg[kSmallMaxE + 1];              // segment starts; seg[E] = rows used
  int warp_cnt[kSmallWarps][kSmallMaxE];
  int warp_sums[kSmallWarps];
  int flags;                            // BSF_DEVERR_* bits seen
};

// Called by all kSmallThreads threads of the CTA.  Fills sm.hist, sm.seg
// (layout: contiguous segments aligned to a_or_m, or masked slots of a_or_m
// rows) and calls on_assign(i, dest) from the thread that owns assignment i,
// dest = packed row or -1 when the assignment is dropped.  Writes no global
// memory itself.
template <class OnAssign>
__device__ __forceinline__ void route_in_block(const int32_t* __restrict__ ids, int64_t R, int E, int layout,
                                               int64_t a_or_m, int64_t m_cap, RouteBlockSmem& sm,
                                               OnAssign&& on_assign) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < E) sm.hist[tid] = 0;
  if (tid == 0) sm.flags = 0;
  __syncthreads();
  for (int64_t i = tid; i < R; i += kSmallThreads) {
    const int id = ids[i];
    if (id >= E) atomicOr(&sm.flags, BSF_DEVERR_EXPERT_ID);
    else if (id >= 0) atomicAdd(&sm.hist[id], 1);
  }
  __syncthreads();
  const int M = tid < E ? sm.hist[tid] : 0;
  if (layout == BSF_LAYOUT_MASKED) {
    if (tid < E) {
      sm.seg[tid] = static_cast<int>(tid * a_or_m);
      if (M > a_or_m) atomicOr(&sm.flags, BSF_DEVERR_MASKED_OVERFLOW);
    }
    if (tid == 0) sm.seg[E] = static_cast<int>(E * a_or_m);
  } else {
    const int len = tid < E ? static_cast<int>((M + a_or_m - 1) / a_or_m * a_or_m) : 0;
    int incl = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sm.warp_sums[warp] = incl;
    __syncthreads();
    int prefix = 0;
    for (int w = 0; w < warp; ++w) prefix += sm.warp_sums[w];
    if (tid < E) {
      sm.seg[tid] = prefix + incl - len;
      if (tid == E - 1) {
        sm.seg[E] = prefix + incl;
        if (prefix + incl > m_cap) atomicOr(&sm.flags, BSF_DEVERR_SEGMENT);
      }
    }
  }
  if (tid < E) sm.base[tid] = 0;
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int64_t r0 = 0; r0 < R; r0 += kSmallThreads) {
    for (int j = tid; j < kSmallWarps * kSmallMaxE; j += kSmallThreads) (&sm.warp_cnt[0][0])[j] = 0;
    __syncthreads();
    const int64_t i = r0 + tid;
    const int id = i < R ? ids[i] : -1;
    const bool valid = id >= 0 && id < E;
    const uint32_t peers = __match_any_sync(0xffffffffu, valid ? id : -1);
    if (valid && (peers & lt_mask) == 0) sm.warp_cnt[warp][id] = __popc(peers);
    __syncthreads();
    if (tid < E) {      // warp-order exclusive prefix on top of the running base
      int run = sm.base[tid];
      for (int w = 0; w < kSmallWarps; ++w) {
        const int c = sm.warp_cnt[w][tid];
        sm.warp_cnt[w][tid] = run;
        run += c;
      }
      sm.base[tid] = run;
    }
    __syncthreads();
    if (i < R) {
      int64_t dest = -1;
      if (valid) {
        const int rank = sm.warp_cnt[warp][id] + __popc(peers & lt_mask);
        if (layout == BSF_LAYOUT_MASKED) {
          if (rank < a_or_m) dest = static_cast<int64_t>(id) * a_or_m + rank;
        } else {
          dest = static_cast<int64_t>(sm.seg[id]) + rank;
        }
        if (dest >= m_cap) {
          dest = -1;
          atomicOr(&sm.flags, BSF_DEVERR_SEGMENT);
        }
      }
      on_assign(i, dest);
    }
    __syncthreads();
  }
}

}  // namespace bsf
