// Deterministic top-k routing: per-expert counts, segment offsets, stable
// ranks, inverse index, and the scatter of quantised rows into the packed
// operand of the grouped GEMM.
//
// "GEMM 执行方式" (rainlin-net) §4.2-§4.3 (topk_ids, M_e, packed rows,
// m_indices, output_index) and §4.6 (A-aligned segments; ep_scatter copies
// each valid route's token and records its row).  "CuTeDSL bei Perplexity",
// MoE dispatch: count tokens per expert, give each a unique index inside its
// expert, then copy rows into (optionally padded) buffers with a wide grid.
//
// Unlike an atomic scatter (whose order inside an expert is arbitrary, §4.6),
// ranks here are stable in the flat assignment index t * k_r + r, so every
// output is bit-reproducible:
//   route_small   count + scan + ranks in one CTA for small batches (decode)
//   route_count   per-chunk expert histograms          (grid: chunks of 512-2048 assignments)
//   route_scan    per-expert prefix over chunks, M_e, aligned segment starts (1 CTA)
//   route_assign  stable ranks -> output_index, token_of_row (grid: chunks)
//   route_fill    per packed row: padding marks, m_indices, row + SF copy (grid: rows)
#include "common.cuh"
#include "host_utils.h"
#include "quant_math.cuh"
#include "route_block.cuh"

namespace bsf {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;  // each warp owns chunk / kWarps consecutive assignments
// Batches of at most kScanInChunks chunks skip route_scan (route_assign_kernel<true>).
constexpr int kScanInChunks = 64;
// Assignments per CTA in count / assign: the smallest of 512, 1024, 2048 that keeps the batch within
// kScanInChunks chunks, else 2048 (with route_scan).  Smaller chunks shorten each CTA's serial
// histogram and rank passes: prefill (32768 assignments) route + quantise-scatter 45.8 -> 38.9 us
// with 512 instead of 2048 (64 vs 16 CTAs), large (65536) 113 -> 108 us with 1024.
constexpr int kChunkMin = 512, kChunkMax = 2048;
inline int route_chunk(int64_t R) {
  int c = kChunkMin;
  while (c < kChunkMax && (R + c - 1) / c > kScanInChunks) c *= 2;
  return c;
}
constexpr int kMaxExperts = 1024;

__global__ void __launch_bounds__(kThreads) route_count_kernel(const int32_t* __restrict__ ids, int64_t R, int E,
                                                               int chunk, int32_t* __restrict__ blk_counts, int* err) {
  pdl_launch_dependents();     // the dependent assign kernel may be scheduled now; it waits for completion
  __shared__ int hist[kMaxExperts];
  __shared__ int bad;
  for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * chunk;
  for (int j = threadIdx.x; j < chunk; j += kThreads) {
    const int64_t i = base + j;
    if (i >= R) break;
    const int id = ids[i];
    if (id >= E) bad = 1;
    else if (id >= 0) atomicAdd(&hist[id], 1);   // counts only: order does not matter
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) blk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
  if (threadIdx.x == 0 && bad) raise_error(err, BSF_DEVERR_EXPERT_ID);
}

// Single CTA of 1024 threads (one expert per thread; E <= 1024).
__global__ void __launch_bounds__(1024) route_scan_kernel(int32_t* __restrict__ blk_counts, int nblk, int E, int layout,
                                                          int64_t align_or_max_m, int64_t m_cap,
                                                          int32_t* __restrict__ counts, int32_t* __restrict__ seg_start,
                                                          int* err) {
  __shared__ int warp_sums[32];
  const int e = threadIdx.x;
  int64_t M = 0;
  if (e < E) {
    for (int b = 0; b < nblk; ++b) {
      const int64_t idx = static_cast<int64_t>(b) * E + e;
      const int c = blk_counts[idx];
      blk_counts[idx] = static_cast<int32_t>(M);   // exclusive prefix over chunks
      M += c;
    }
  }
  if (layout == BSF_LAYOUT_MASKED) {
    if (e < E) {
      const int64_t placed = M < align_or_max_m ? M : align_or_max_m;
      counts[e] = static_cast<int32_t>(placed);
      seg_start[e] = static_cast<int32_t>(e * align_or_max_m);
      if (M > align_or_max_m) raise_error(err, BSF_DEVERR_MASKED_OVERFLOW);
    }
    if (e == 0) seg_start[E] = static_cast<int32_t>(E * align_or_max_m);
    return;
  }
  // contiguous: exclusive scan of the aligned segment lengths over experts
  const int64_t len = e < E ? (M + align_or_max_m - 1) / align_or_max_m * align_or_max_m : 0;
  int64_t incl = len;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = static_cast<int>(incl);
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += v;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int64_t warp_prefix = warp > 0 ? warp_sums[warp - 1] : 0;
  const int64_t excl = warp_prefix + incl - len;
  if (e < E) {
    counts[e] = static_cast<int32_t>(M);
    seg_start[e] = static_cast<int32_t>(excl);
  }
  if (e == E - 1) {
    seg_start[E] = static_cast<int32_t>(excl + len);
    if (excl + len > m_cap) raise_error(err, BSF_DEVERR_SEGMENT);
  }
}

// Batches of at most kScanInChunks chunks skip route_scan: every assign CTA reads all chunks'
// histograms (nblk x E words, from L2) and derives its own chunk's per-expert base, the counts and
// the segment starts itself, with the same integer arithmetic as route_scan; CTA 0 stores counts and
// seg_start.  One launch fewer (route_scan ran as a single CTA).

// All threads of the CTA.  blk = raw per-chunk histograms [nblk][E]; fills base[e] (assignments of
// expert e in chunks before `b`), tot[e] (M_e) and seg[0..E] (contiguous: aligned exclusive scan of
// M_e; masked: slots of max_m rows); returns BSF_DEVERR_* bits seen (CTA-uniform).
__device__ int scan_chunks(const int32_t* __restrict__ blk, int nblk, int b, int E, int layout, int64_t a_or_m,
                           int64_t m_cap, int* base, int* tot, int* seg, int* warp_sums) {
  __shared__ int bad;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) bad = 0;
  for (int e = tid; e < E; e += kThreads) {
    int pre = 0, sum = 0;
    for (int bb = 0; bb < nblk; ++bb) {
      const int c = blk[static_cast<int64_t>(bb) * E + e];
      if (bb < b) pre += c;
      sum += c;
    }
    base[e] = pre;
    tot[e] = sum;
  }
  __syncthreads();
  if (layout == BSF_LAYOUT_MASKED) {
    for (int e = tid; e < E; e += kThreads) {
      seg[e] = static_cast<int>(e * a_or_m);
      if (tot[e] > a_or_m) bad = BSF_DEVERR_MASKED_OVERFLOW;
    }
    if (tid == 0) seg[E] = static_cast<int>(E * a_or_m);
    __syncthreads();
    return bad;
  }
  // contiguous: thread tid owns experts 4 tid .. 4 tid + 3 (E <= 1024 = 4 x kThreads)
  int64_t len[4], own = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * tid + j;
    len[j] = e < E ? (tot[e] + a_or_m - 1) / a_or_m * a_or_m : 0;
    own += len[j];
  }
  int64_t incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = static_cast<int>(incl);
  __syncthreads();
  int64_t run = incl - own;
  for (int w = 0; w < warp; ++w) run += warp_sums[w];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * tid + j;
    if (e < E) seg[e] = static_cast<int>(run);
    run += len[j];
    if (e == E - 1) {
      seg[E] = static_cast<int>(run);
      if (run > m_cap) bad = BSF_DEVERR_SEGMENT;
    }
  }
  __syncthreads();
  return bad;
}

// SCAN = false: blk holds each chunk's exclusive per-expert prefix (route_scan's output) and
// seg_start the segment starts.  SCAN = true: blk holds the raw per-chunk histograms; the CTA derives
// both itself (scan_chunks) and CTA 0 writes counts and seg_start.
template <bool SCAN>
__global__ void __launch_bounds__(kThreads) route_assign_kernel(const int32_t* __restrict__ ids, int64_t R, int kr,
                                                                int E, int layout, int64_t max_m, int64_t m_cap,
                                                                const int32_t* __restrict__ blk_base, int nblk,
                                                                int chunk,
                                                                int32_t* __restrict__ seg_start,
                                                                int32_t* __restrict__ counts,
                                                                int32_t* __restrict__ output_index,
                                                                int32_t* __restrict__ token_of_row,
                                                                int32_t* __restrict__ m_indices, int mark_rows,
                                                                int* err) {
  // launched as a programmatic dependent: nothing the preceding kernel writes is read before this
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int smem[];
  int* warp_cnt = smem;                       // [kWarps][E]
  int* seg = smem + kWarps * E;               // [E + 1]
  int* base = seg + E + 1;                    // [E] (SCAN)
  int* tot = base + E;                        // [E] (SCAN)
  __shared__ int overflow;
  __shared__ int warp_sums[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = threadIdx.x; j < kWarps * E; j += kThreads) warp_cnt[j] = 0;
  if (threadIdx.x == 0) overflow = 0;
  if constexpr (SCAN) {
    const int bad = scan_chunks(blk_base, nblk, static_cast<int>(blockIdx.x), E, layout, max_m, m_cap, base, tot, seg,
                                warp_sums);
    if (blockIdx.x == 0) {
      for (int e = threadIdx.x; e < E; e += kThreads) {
        counts[e] = layout == BSF_LAYOUT_MASKED ? (tot[e] < max_m ? tot[e] : static_cast<int>(max_m)) : tot[e];
        seg_start[e] = seg[e];
      }
      if (threadIdx.x == 0) {
        seg_start[E] = seg[E];
        if (bad) raise_error(err, bad);
      }
    }
    if (mark_rows) {
      // padding rows of experts e = b, b + grid, ...: token -1, owner e (what route_fill does without
      // a scatter source, so that no fill launch is needed)
      for (int e = blockIdx.x; e < E; e += gridDim.x) {
        const int placed = layout == BSF_LAYOUT_MASKED ? (tot[e] < max_m ? tot[e] : static_cast<int>(max_m)) : tot[e];
        const int64_t end = layout == BSF_LAYOUT_MASKED ? static_cast<int64_t>(seg[e]) + max_m : seg[e + 1];
        for (int64_t r = static_cast<int64_t>(seg[e]) + placed + threadIdx.x; r < end && r < m_cap; r += kThreads) {
          token_of_row[r] = -1;
          if (m_indices) m_indices[r] = e;
        }
      }
    }
  } else {
    for (int e = threadIdx.x; e < E; e += kThreads) seg[e] = seg_start[e];
  }
  __syncthreads();

  const int sub = chunk / kWarps;             // this warp's consecutive assignments (64 .. 256)
  const int64_t sub0 = static_cast<int64_t>(blockIdx.x) * chunk + warp * sub;
  const uint32_t lt_mask = (1u << lane) - 1u;
  // pass 1: per-warp histogram of its sub-chunk
  for (int r = 0; r < sub; r += 32) {
    const int64_t i = sub0 + r + lane;
    int id = i < R ? ids[i] : -1;
    const bool valid = id >= 0 && id < E;
    const int key = valid ? id : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    if (valid && (peers & lt_mask) == 0) warp_cnt[warp * E + id] += __popc(peers);
  }
  __syncthreads();
  // exclusive prefix over the warps, on top of this chunk's base per expert
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int run = SCAN ? base[e] : blk_base[static_cast<int64_t>(blockIdx.x) * E + e];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = warp_cnt[w * E + e];
      warp_cnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // pass 2: stable rank = warp base + earlier matches in this warp's sub-chunk
  for (int r = 0; r < sub; r += 32) {
    const int64_t i = sub0 + r + lane;
    const int id = i < R ? ids[i] : -1;
    const bool valid = id >= 0 && id < E;
    const int key = valid ? id : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    int rank = 0;
    if (valid) rank = warp_cnt[warp * E + id] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) warp_cnt[warp * E + id] += __popc(peers);
    __syncwarp();
    if (i < R) {
      int64_t dest = -1;
      if (valid) {
        if (layout == BSF_LAYOUT_MASKED) {
          if (rank < max_m) dest = static_cast<int64_t>(id) * max_m + rank;
        } else {
          dest = static_cast<int64_t>(seg[id]) + rank;
        }
        if (dest >= m_cap) {
          dest = -1;
          overflow = 1;
        }
      }
      output_index[i] = static_cast<int32_t>(dest);
      if (dest >= 0) {
        token_of_row[dest] = static_cast<int32_t>(i / kr);
        if (SCAN && mark_rows && m_indices) m_indices[dest] = id;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && overflow) raise_error(err, BSF_DEVERR_SEGMENT);
}

// Small batches (decode): one CTA routes the whole batch (route_block.cuh).
__global__ void __launch_bounds__(kSmallThreads) route_small_kernel(const int32_t* __restrict__ ids, int64_t R,
                                                                    int kr, int E, int layout, int64_t a_or_m,
                                                                    int64_t m_cap, int32_t* __restrict__ counts,
                                                                    int32_t* __restrict__ seg_start,
                                                                    int32_t* __restrict__ output_index,
                                                                    int32_t* __restrict__ token_of_row, int* err) {
  pdl_launch_dependents();     // the dependent fill kernel may be scheduled now; it waits for completion
  __shared__ RouteBlockSmem sm;
  route_in_block(ids, R, E, layout, a_or_m, m_cap, sm, [&](int64_t i, int64_t dest) {
    output_index[i] = static_cast<int32_t>(dest);
    if (dest >= 0) token_of_row[dest] = static_cast<int32_t>(i / kr);
  });
  const int tid = threadIdx.x;
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

constexpr int kFillRows = 32;   // packed rows per CTA in route_fill

// Per packed row r < seg_start[E]: mark padding rows (token -1), write
// m_indices, and copy a routed row's data (row_bytes, FP8 or NVFP4) and its
// n_words SF words.
__global__ void __launch_bounds__(kThreads) route_fill_kernel(int E, int64_t m_cap, const int32_t* __restrict__ counts,
                                                              const int32_t* __restrict__ seg_start,
                                                              int32_t* __restrict__ token_of_row,
                                                              int32_t* __restrict__ m_indices,
                                                              const uint8_t* __restrict__ q,
                                                              const int32_t* __restrict__ sf, int64_t sf_ld,
                                                              int64_t row_bytes, int64_t n_words,
                                                              uint8_t* __restrict__ a_packed,
                                                              int32_t* __restrict__ sfa_packed, int64_t sfa_ld) {
  pdl_launch_dependents();     // a dependent GEMM may be scheduled now; it waits for completion
  pdl_wait();                  // launched as a dependent of the routing kernel: its outputs are complete
  __shared__ int tok[kFillRows];
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kFillRows;
  const int64_t rows_used = seg_start[E];
  if (row0 >= rows_used || row0 >= m_cap) return;
  if (threadIdx.x < kFillRows) {
    const int64_t r = row0 + threadIdx.x;
    int t = -2;                                  // -2: outside the used rows
    if (r < rows_used && r < m_cap) {
      int lo = 0, hi = E - 1;                    // last expert with seg_start[e] <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg_start[mid] <= r) lo = mid; else hi = mid - 1;
      }
      // skip empty segments that share the start
      const bool pad = r - seg_start[lo] >= counts[lo];
      if (pad) {
        token_of_row[r] = -1;
        t = -1;
      } else {
        t = token_of_row[r];
      }
      if (m_indices) m_indices[r] = lo;
    }
    tok[threadIdx.x] = t;
  }
  __syncthreads();
  if (q == nullptr) return;
  // SF words of routed rows: thread (word i, row) with consecutive rows -> coalesced stores.
  // Padding rows keep whatever the buffer held: "GEMM 执行方式" §4.6 leaves them
  // uninitialised, and no computed output row depends on them.
  for (int64_t j = threadIdx.x; j < n_words * kFillRows; j += kThreads) {
    const int64_t i = j / kFillRows;
    const int rl = static_cast<int>(j % kFillRows);
    const int t = tok[rl];
    if (t < 0) continue;
    sfa_packed[i * sfa_ld + row0 + rl] = sf[i * sf_ld + t];
  }
  // data rows: one warp per routed row, 16-byte vectors
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nvec = row_bytes / 16;
  for (int rl = warp; rl < kFillRows; rl += kWarps) {
    const int t = tok[rl];
    if (t < 0) continue;
    uint4* dst = reinterpret_cast<uint4*>(a_packed + (row0 + rl) * row_bytes);
    const uint4* src = reinterpret_cast<const uint4*>(q + static_cast<int64_t>(t) * row_bytes);
    for (int64_t v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
  }
}

// bsf_route_quantise: one warp per (token t, 512-wide K group g).  The token's bf16 row segment is
// read once, quantised with the arithmetic of quantise_act_kernel (quant_math.cuh, so the bytes are
// the same), and its E4M3 codes and scale word are written to each of the token's k_r packed rows
// (output_index from the assign kernel; -1 = dropped).  Launched as a programmatic dependent of the
// routing kernels: the loads of x and the quantisation run before the wait (x is complete before the
// count kernel, a plain launch, starts; the assign kernel triggers this launch only after the count
// kernel has completed), the reads of output_index and the stores after it.
__global__ void __launch_bounds__(kThreads) quantise_scatter_kernel(const uint16_t* __restrict__ x, int64_t T,
                                                                    int64_t K, int kr,
                                                                    const int32_t* __restrict__ output_index,
                                                                    uint8_t* __restrict__ a_packed,
                                                                    int32_t* __restrict__ sfa_packed, int64_t sfa_ld) {
  pdl_launch_dependents();     // a dependent GEMM may be scheduled now; it waits for completion
  const int64_t n_groups = (K + 511) / 512;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const bool in_range = gw < T * n_groups;        // warp-uniform
  const int64_t t = in_range ? gw / n_groups : 0;
  const int64_t g = in_range ? gw - t * n_groups : 0;
  const int64_t k0 = g * 512 + lane * 16;
  const bool active = in_range && k0 < K;
  uint4 ra = make_uint4(0, 0, 0, 0), rb = ra;
  if (active) {                                   // x is not written by the routing kernels
    const uint4* src = reinterpret_cast<const uint4*>(x + t * K + k0);
    ra = __ldg(src);
    rb = __ldg(src + 1);
  }
  if (!in_range) {
    pdl_wait();
    return;
  }
  float v[16];
  float amax = 0.f;
  if (active) {
    float fa[8], fb[8];
    bf16x8_to_float(ra, fa);
    bf16x8_to_float(rb, fb);
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
  uint4 out = make_uint4(0, 0, 0, 0);
  if (active) {
    const float s = inv_pow2(e);
    out.x = pack4_e4m3(v[0] * s, v[1] * s, v[2] * s, v[3] * s);
    out.y = pack4_e4m3(v[4] * s, v[5] * s, v[6] * s, v[7] * s);
    out.z = pack4_e4m3(v[8] * s, v[9] * s, v[10] * s, v[11] * s);
    out.w = pack4_e4m3(v[12] * s, v[13] * s, v[14] * s, v[15] * s);
  }
  // byte j of the SF word = block j of the group (127 for blocks past K)
  const uint32_t byte = active ? static_cast<uint32_t>(e + 127) : 127u;
  const uint32_t b0 = __shfl_sync(0xffffffffu, byte, 0);
  const uint32_t b1 = __shfl_sync(0xffffffffu, byte, 8);
  const uint32_t b2 = __shfl_sync(0xffffffffu, byte, 16);
  const uint32_t b3 = __shfl_sync(0xffffffffu, byte, 24);
  const int32_t word = static_cast<int32_t>(b0 | (b1 << 8) | (b2 << 16) | (b3 << 24));
  // the quantisation above needs nothing from the routing kernels; only the destinations do
  pdl_wait();                                     // output_index is complete
  const int dest_l = lane < kr ? output_index[t * kr + lane] : -1;
  for (int r = 0; r < kr; ++r) {
    const int dest = __shfl_sync(0xffffffffu, dest_l, r);   // warp-uniform
    if (dest < 0) continue;
    if (active) *reinterpret_cast<uint4*>(a_packed + static_cast<int64_t>(dest) * K + k0) = out;
    if (lane == 0) sfa_packed[g * sfa_ld + dest] = word;
  }
}

}  // namespace
}  // namespace bsf

using namespace bsf;

extern "C" size_t bsf_route_workspace_bytes(int64_t T, int64_t kr, int64_t E) {
  if (T < 0 || kr <= 0 || E <= 0 || T > INT32_MAX / kr) return 0;   // T * kr is formed only when it fits
  const int64_t R = T * kr;
  const int chunk = route_chunk(R);
  const int64_t nblk = (R + chunk - 1) / chunk;
  return static_cast<size_t>((nblk > 0 ? nblk : 1) * E * sizeof(int32_t));
}

namespace bsf {
namespace {

enum RowFormat { kRowsFp8, kRowsNvfp4, kRowsBf16, kRowsFp8F32 };

// bsf_route / bsf_route_nvfp4 / bsf_route_bf16: fmt selects the scatter's row format
// (FP8: K bytes + ceil(K/512) SF words; NVFP4: K/2 bytes + K/64 words; BF16: 2K bytes, no SF).
bsf_status route_impl(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout, int64_t align_or_max_m,
                      int32_t* counts, int32_t* seg_start, int32_t* output_index, int32_t* token_of_row,
                      int32_t* m_indices, int64_t m_cap, const uint8_t* q, const int32_t* sf, int64_t sf_ld,
                      int64_t K, RowFormat fmt, uint8_t* a_packed, int32_t* sfa_packed, int64_t sfa_ld,
                      void* workspace, size_t workspace_bytes, bsf_stream_t stream) {
  if (T < 0 || kr <= 0 || E <= 0 || E > kMaxExperts) return BSF_ERR_INVALID_ARGUMENT;
  if (layout != BSF_LAYOUT_CONTIGUOUS && layout != BSF_LAYOUT_MASKED) return BSF_ERR_INVALID_ARGUMENT;
  if (align_or_max_m < 1 || align_or_max_m > INT32_MAX) return BSF_ERR_INVALID_ARGUMENT;
  if (!counts || !seg_start || !output_index || !token_of_row) return BSF_ERR_INVALID_ARGUMENT;
  if (T > INT32_MAX / kr) return BSF_ERR_UNSUPPORTED;   // before forming R, which must not wrap
  const int64_t R = T * kr;
  const int64_t need_cap = layout == BSF_LAYOUT_MASKED ? E * align_or_max_m : R + E * (align_or_max_m - 1);
  if (m_cap < need_cap || m_cap > INT32_MAX) return BSF_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < bsf_route_workspace_bytes(T, kr, E) || !workspace) return BSF_ERR_INVALID_ARGUMENT;
  if (q && fmt == kRowsBf16) {
    if (!a_packed || K <= 0 || K % 8) return BSF_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(a_packed)) return BSF_ERR_MISALIGNED;
  } else if (q) {
    if (!sf || !a_packed || !sfa_packed || K <= 0 || K % (fmt == kRowsNvfp4 ? 64 : 128))
      return BSF_ERR_INVALID_ARGUMENT;
    if (sf_ld < T || sf_ld % 4 || sfa_ld < m_cap || sfa_ld % 4) return BSF_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(a_packed) || !aligned16(sf) || !aligned16(sfa_packed)) return BSF_ERR_MISALIGNED;
  }
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int chunk = route_chunk(R);
  const int nblk = static_cast<int>((R + chunk - 1) / chunk);
  int32_t* blk = static_cast<int32_t*>(workspace);
  const int e32 = static_cast<int>(E);
  bool marks_in_assign = false;
  if (R <= kSmallMaxR && E <= kSmallMaxE) {
    route_small_kernel<<<1, kSmallThreads, 0, s>>>(topk_ids, R, static_cast<int>(kr), e32, layout, align_or_max_m,
                                                   m_cap, counts, seg_start, output_index, token_of_row, err);
  } else {
    if (nblk > 0) {
      route_count_kernel<<<nblk, kThreads, 0, s>>>(topk_ids, R, e32, chunk, blk, err);
    }
    bsf_status st = BSF_OK;
    if (nblk <= kScanInChunks) {
      // (R = 0: one CTA only writes the counts and segment starts).  Without a scatter source the
      // assign CTAs also mark the padding rows and write m_indices, and no fill kernel follows.
      marks_in_assign = q == nullptr;
      const size_t smem = (static_cast<size_t>(kWarps + 3) * E + 1) * sizeof(int);
      st = launch_dependent(route_assign_kernel<true>, static_cast<unsigned>(nblk > 0 ? nblk : 1), kThreads, smem, s,
                            topk_ids, R, static_cast<int>(kr), e32, layout, align_or_max_m, m_cap,
                            static_cast<const int32_t*>(blk), nblk, chunk, seg_start, counts, output_index,
                            token_of_row, m_indices, static_cast<int>(marks_in_assign), err);
    } else {
      route_scan_kernel<<<1, 1024, 0, s>>>(blk, nblk, e32, layout, align_or_max_m, m_cap, counts, seg_start, err);
      const size_t smem = (static_cast<size_t>(kWarps + 1) * E + 1) * sizeof(int);
      st = launch_dependent(route_assign_kernel<false>, static_cast<unsigned>(nblk), kThreads, smem, s, topk_ids, R,
                            static_cast<int>(kr), e32, layout, align_or_max_m, m_cap,
                            static_cast<const int32_t*>(blk), nblk, chunk, seg_start, counts, output_index,
                            token_of_row, m_indices, 0, err);
    }
    if (st != BSF_OK) return st;
  }
  const int64_t fill_blocks = marks_in_assign ? 0 : (m_cap + kFillRows - 1) / kFillRows;
  if (fill_blocks > 0) {
    const bsf_status st = launch_dependent(
        route_fill_kernel, static_cast<unsigned>(fill_blocks), kThreads, 0, s, e32, m_cap,
        static_cast<const int32_t*>(counts), static_cast<const int32_t*>(seg_start), token_of_row, m_indices, q, sf,
        sf_ld, fmt == kRowsNvfp4 ? K / 2 : fmt == kRowsBf16 ? 2 * K : K,
        fmt == kRowsNvfp4 ? K / 64 : fmt == kRowsBf16 ? 0 : fmt == kRowsFp8F32 ? K / 128 : (K + 511) / 512, a_packed,
        sfa_packed, sfa_ld);
    if (st != BSF_OK) return st;
  }
  return launch_status();
}

}  // namespace
}  // namespace bsf

extern "C" bsf_status bsf_route(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout,
                                int64_t align_or_max_m, int32_t* counts, int32_t* seg_start, int32_t* output_index,
                                int32_t* token_of_row, int32_t* m_indices, int64_t m_cap, const uint8_t* q,
                                const int32_t* sf, int64_t sf_ld, int64_t K, uint8_t* a_packed, int32_t* sfa_packed,
                                int64_t sfa_ld, void* workspace, size_t workspace_bytes, bsf_stream_t stream) {
  return route_impl(topk_ids, T, kr, E, layout, align_or_max_m, counts, seg_start, output_index, token_of_row,
                    m_indices, m_cap, q, sf, sf_ld, K, kRowsFp8, a_packed, sfa_packed, sfa_ld, workspace,
                    workspace_bytes, stream);
}

extern "C" bsf_status bsf_route_nvfp4(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout,
                                      int64_t align_or_max_m, int32_t* counts, int32_t* seg_start,
                                      int32_t* output_index, int32_t* token_of_row, int32_t* m_indices,
                                      int64_t m_cap, const uint8_t* q, const int32_t* sf, int64_t sf_ld, int64_t K,
                                      uint8_t* a_packed, int32_t* sfa_packed, int64_t sfa_ld, void* workspace,
                                      size_t workspace_bytes, bsf_stream_t stream) {
  return route_impl(topk_ids, T, kr, E, layout, align_or_max_m, counts, seg_start, output_index, token_of_row,
                    m_indices, m_cap, q, sf, sf_ld, K, kRowsNvfp4, a_packed, sfa_packed, sfa_ld, workspace,
                    workspace_bytes, stream);
}

extern "C" bsf_status bsf_route_f32sf(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout,
                                      int64_t align_or_max_m, int32_t* counts, int32_t* seg_start,
                                      int32_t* output_index, int32_t* token_of_row, int32_t* m_indices,
                                      int64_t m_cap, const uint8_t* q, const float* sf, int64_t sf_ld, int64_t K,
                                      uint8_t* a_packed, float* sfa_packed, int64_t sfa_ld, void* workspace,
                                      size_t workspace_bytes, bsf_stream_t stream) {
  return route_impl(topk_ids, T, kr, E, layout, align_or_max_m, counts, seg_start, output_index, token_of_row,
                    m_indices, m_cap, q, reinterpret_cast<const int32_t*>(sf), sf_ld, K, kRowsFp8F32, a_packed,
                    reinterpret_cast<int32_t*>(sfa_packed), sfa_ld, workspace, workspace_bytes, stream);
}

extern "C" bsf_status bsf_route_bf16(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout,
                                     int64_t align_or_max_m, int32_t* counts, int32_t* seg_start,
                                     int32_t* output_index, int32_t* token_of_row, int32_t* m_indices, int64_t m_cap,
                                     const void* x, int64_t K, void* a_packed, void* workspace,
                                     size_t workspace_bytes, bsf_stream_t stream) {
  return route_impl(topk_ids, T, kr, E, layout, align_or_max_m, counts, seg_start, output_index, token_of_row,
                    m_indices, m_cap, static_cast<const uint8_t*>(x), nullptr, 0, K, kRowsBf16,
                    static_cast<uint8_t*>(a_packed), nullptr, 0, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of bsf_route.
//
// For callers that cannot call cudaMalloc where they route: serving runtimes
// that reserve all device memory at start-up (an allocation would fail or
// fragment their pool, and cudaMalloc synchronises the device), plug-ins whose
// host framework owns the allocator, and code inside an allocator callback.
// The per-chunk expert counts live in a fixed file-scope device array instead
// of a caller-provided workspace.
namespace bsf {
namespace {

constexpr size_t kRouteStaticScratchBytes = BSF_ROUTE_STATIC_SCRATCH_BYTES;

// Shared by every call on a device; every GPU that loads the library holds it until exit.
static __device__ __align__(256) int32_t g_route_scratch[kRouteStaticScratchBytes / sizeof(int32_t)];

// Device address of g_route_scratch for the current device, resolved once per
// device with that device current (the host-side name is only a stand-in).
// The cache entries are atomics: first calls from several host threads may
// race to fill an entry, and each stores the same address.
int32_t* route_scratch_ptr(bsf_status* st) {
  static std::atomic<int32_t*> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *st = BSF_ERR_CUDA;
    return nullptr;
  }
  int32_t* ptr = cached[dev].load(std::memory_order_acquire);
  if (ptr == nullptr) {
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_route_scratch) != cudaSuccess || ptr == nullptr) {
      *st = BSF_ERR_CUDA;
      return nullptr;
    }
    cached[dev].store(ptr, std::memory_order_release);
  }
  *st = BSF_OK;
  return ptr;
}

}  // namespace
}  // namespace bsf

extern "C" bsf_status bsf_route_no_alloc(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout,
                                         int64_t align_or_max_m, int32_t* counts, int32_t* seg_start,
                                         int32_t* output_index, int32_t* token_of_row, int32_t* m_indices,
                                         int64_t m_cap, const uint8_t* q, const int32_t* sf, int64_t sf_ld,
                                         int64_t K, uint8_t* a_packed, int32_t* sfa_packed, int64_t sfa_ld,
                                         bsf_stream_t stream) {
  if (T < 0 || kr <= 0 || E <= 0) return BSF_ERR_INVALID_ARGUMENT;
  if (T > INT32_MAX / kr) return BSF_ERR_UNSUPPORTED;
  const size_t need = bsf_route_workspace_bytes(T, kr, E);
  if (need > kRouteStaticScratchBytes) return BSF_ERR_UNSUPPORTED;   // problem larger than the static scratch
  bsf_status st = BSF_OK;
  int32_t* scratch = route_scratch_ptr(&st);
  if (st != BSF_OK) return st;
  // The count kernel overwrites every scratch word the later kernels read, so
  // the previous call's contents need no clearing.
  return bsf_route(topk_ids, T, kr, E, layout, align_or_max_m, counts, seg_start, output_index, token_of_row,
                   m_indices, m_cap, q, sf, sf_ld, K, a_packed, sfa_packed, sfa_ld, scratch, kRouteStaticScratchBytes,
                   stream);
}

extern "C" bsf_status bsf_route_quantise(const void* x, int64_t T, int64_t K, const int32_t* topk_ids, int64_t kr,
                                         int64_t E, int layout, int64_t align_or_max_m, int32_t* counts,
                                         int32_t* seg_start, int32_t* output_index, int32_t* token_of_row,
                                         int32_t* m_indices, int64_t m_cap, uint8_t* a_packed, int32_t* sfa_packed,
                                         int64_t sfa_ld, void* workspace, size_t workspace_bytes,
                                         bsf_stream_t stream) {
  if (!x || !a_packed || !sfa_packed || K <= 0 || K % 128) return BSF_ERR_INVALID_ARGUMENT;
  if (kr > 32) return BSF_ERR_UNSUPPORTED;      // one lane per assignment of a token
  if (sfa_ld < m_cap || sfa_ld % 4) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(a_packed) || !aligned16(sfa_packed)) return BSF_ERR_MISALIGNED;
  if (!fits_rows(T, K)) return BSF_ERR_UNSUPPORTED;
  // routing, segment starts, padding marks and m_indices: bsf_route without a scatter source
  bsf_status st = bsf_route(topk_ids, T, kr, E, layout, align_or_max_m, counts, seg_start, output_index, token_of_row,
                            m_indices, m_cap, nullptr, nullptr, 0, K, nullptr, nullptr, 0, workspace, workspace_bytes,
                            stream);
  if (st != BSF_OK || T == 0) return st;
  const int64_t warps = T * ((K + 511) / 512);
  const int64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
  if (blocks > INT32_MAX) return BSF_ERR_UNSUPPORTED;
  return launch_dependent(quantise_scatter_kernel, static_cast<unsigned>(blocks), kThreads, 0,
                          reinterpret_cast<cudaStream_t>(stream), static_cast<const uint16_t*>(x), T, K,
                          static_cast<int>(kr), static_cast<const int32_t*>(output_index), a_packed, sfa_packed,
                          sfa_ld);
}
