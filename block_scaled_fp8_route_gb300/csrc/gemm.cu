// Grouped FP8 block-scaled GEMM over per-expert token segments, sm_103a.
//
//   D[r, n] = BF16( sum_k A[r, k] sA[r, k/128] * B_e[n, k] sB_e[n/128, k/128] )
//   for every expert e and row r of its segment.
//
// Sources: "GEMM 执行方式" §4.1 (P independent problems), §4.4 (Y_e = X_e W_e^T);
// "AsymGEMM" README ("K-outer, M-inner Loop": a weight tile is fetched once
// and reused for all token tiles of its expert; "asymScheduler": CTAs own
// (N-tile, expert) work with no atomics; "Token Layout Protocols");
// DeepGEMM FP8 article "补偿机制二" (the tensor core applies the UE8M0 block
// scales itself, selected by a scale-factor id in the instruction descriptor).
//
// GB300 design (not the pages' kernels):
// * swap-AB: the MMA's M = 128 rows are WEIGHT rows (an N-tile of the output)
//   and the MMA's N dimension is the expert's TOKENS (16..256, step 16), so
//   a segment of 8 tokens costs a 128 x 16 MMA instead of a padded 128 x 128;
// * persistent CTAs (one or two per SM); work item = (expert, N-tile, token
//   chunk), chunks fastest so concurrent CTAs share the weight tile in L2;
//   large FP8 batches take 256-row items (two 128-row weight tiles sharing
//   one token chunk, one MMA per weight tile per K-step);
// * warp roles: warp 0 TMA producer, warp 1 MMA issuer + TMEM owner,
//   warps 2-5 epilogue, warps 6-9 scale-factor loaders (256-row items:
//   warps 10-13 a second epilogue group, warp 14 the waiter that performs the
//   issuers' mbarrier waits, warp 15 a second MMA issuer);
// * weights either row-major [E, N, K] or tiled (each 128 x 128-byte TMA box
//   one contiguous 16 KB run, BSF_B_TILED);
// * operands: K-major, 128-byte swizzled tiles of 128 K (TMA), STAGES-deep
//   mbarrier ring; accumulator 128 lanes x TOK fp32 columns in TMEM;
// * scales: kind::mxf8f6f4 block scaling with one UE8M0 per row per 32 K;
//   our 128-wide blocks use one byte for all four K-steps of a block: the
//   int32 word holding four consecutive blocks is written to TMEM once per
//   512 K and the byte is picked with sf_id = k_block % 4;
// * epilogue: tcgen05.ld 32 columns (tokens) per thread row (weight row); after
//   one exchange between neighbour lanes each lane stores two weight rows of one
//   token (4 bytes), a warp's store covering two tokens' 64-byte row segments of D.
#include "common.cuh"
#include "host_utils.h"
#include "tma_map.h"

namespace bsf {

namespace {

constexpr int kBlockW = 128;        // weight rows per tile (MMA M)
constexpr int kBlockK = 128;        // K per pipeline stage (one 128-byte swizzle row of FP8)
constexpr int kMaxExperts = 1024;
constexpr int kBigTok = 224;        // token tile of the large-segment variant
constexpr int kWideTok = 160;       // token chunk of the four-stage 256-row items (at most 256 experts)
constexpr int kHostTok = 448;       // token tile of the host-weight (K-outer / M-inner) variant
constexpr int kFmtFp8 = 0;          // E4M3 operands, UE8M0 scales per 128 K (kind::mxf8f6f4, 1X)
constexpr int kFmtNvfp4 = 1;        // E2M1 operands, UE4M3 scales per 16 K (kind::mxf4nvf4, 4X)
constexpr int kFmtBf16 = 2;         // BF16 operands, no scales (kind::f16)
constexpr int kFmtFp8F32 = 3;       // E4M3 operands, float32 scales applied in software per 128-K block
constexpr int kNvfp4MaxE = 256;     // NVFP4 variants size their tile tables for 256 experts
constexpr int kPrefetchStages = 12; // weight stages a dependent small-batch CTA pulls into L2 before its wait

struct GemmArgs {
  const int32_t* seg_start;  // contiguous: [E+1]; masked: nullptr
  const int32_t* counts;     // rows per expert (counts / masked_m)
  int64_t max_m;             // masked slot stride (0 for contiguous)
  int64_t m_rows;            // rows of A and D
  const int32_t* sfa;
  int64_t sfa_ld;
  const int32_t* sfb;        // [E][nw][N]
  uint16_t* d;
  int E, N, K;
  int* err;
  int flags;                 // BSF_B_TILED (weight layout), BSF_DEBUG_WITHHOLD_LOADS (test-only fault injection)
  int a_exp;                 // NVFP4: tensor exponent of A
  const int32_t* b_exp;      // NVFP4: tensor exponent per expert of B [E]
  const float* sfa_f32;      // FP32 scales: A [K/128][sfa_ld]
  const float* sfb_f32;      // FP32 scales: B [E][N/128][K/128]
};

// TOK = token columns of one tile's accumulator.  64 and 224 keep two
// accumulators in TMEM so the epilogue of one tile overlaps the MMAs of the
// next (2 x 64 + 4 x 8 SF columns; 2 x 224 + 4 x 16 = 512).  448 holds all
// tokens of an expert (up to 448) in one accumulator, issued as two MMAs of
// N <= 224 per K-step, so each weight tile is fetched once and reused for all
// of them (the K-outer / M-inner order of the "AsymGEMM" README; used when the
// weights live in host memory and every re-fetch crosses the host link).
// CPS = CTAs resident per SM.  With CPS = 2 each CTA keeps one accumulator
// and half the ring, and the two CTAs' single-thread MMA issuers share the
// SM's tensor core, so one CTA's barrier waits and epilogue drain are covered
// by the other's MMAs.
// MAXE = the most experts the per-CTA tile tables hold; the small-batch tile with at most 256
// experts turns the table space it saves into a fourth pipeline stage (-1.4 % at decode).
// FMT = operand format.  A stage is always 128 bytes of K per row: 128 FP8
// values (four K = 32 MMAs) or 256 NVFP4 values (four K = 64 MMAs).  FP8
// scale words cover four stages (one byte per stage, picked by sf_id);
// NVFP4 needs a word per row per MMA, so its SF slot covers one stage:
// 4 x 4 weight columns + 4 x 4 token columns (tokens <= 128).
// WT = weight tiles per work item.  WT = 2 (FP8 or BF16, 224 tokens, one CTA per SM): a stage holds two
// 128-row weight tiles and one token tile, and each K-step issues one MMA per weight tile into its
// own 224-column accumulator, so a work item is a 256 x 224 output block.  The bytes a stage brings
// into shared memory then cover 1.47x the MMA work of the 128 x 224 tile ((256 + 224) bytes per
// 256 x 224 products against (128 + 224) per 128 x 224), which is what a latency-bound load
// pipeline needs; the price is that the epilogue of one item no longer overlaps the next item's MMAs.
// With at most 256 experts the items are 256 x 160 (kWideTok) instead: the smaller token tile and
// the smaller tile tables make room for a fourth stage, and
// with the load pipeline the limit (two MMA issuers keep the tensor core fed) the extra stage in
// flight pays: same-box A/B, FP8 large gate-up 1713 -> 1534 us, large down 1020 -> 882 us, prefill
// gate-up 378 -> 367 us; BF16 large gate-up 3160 -> 2826 us; outputs bit-identical.
template <int TOK, int CPS = 1, int MAXE = kMaxExperts, int FMT = kFmtFp8, int WT = 1>
struct Cfg {
  static constexpr bool kFp4 = FMT == kFmtNvfp4;
  static constexpr bool kBf16 = FMT == kFmtBf16;            // no scale factors: SF warps idle
  // float32 scales: each 128-K stage is multiplied into its own TMEM partial (two buffers),
  // which the epilogue warps scale and add into registers (the SF warps idle)
  static constexpr bool kF32 = FMT == kFmtFp8F32;
  static constexpr int kMaxE = MAXE;
  static constexpr int kKElems = kFp4 ? 256 : kBf16 ? 64 : 128;   // K values per stage
  static constexpr int kKbPerSlot = kFp4 ? 1 : 4;            // stages per SF slot
  // NVFP4 stages also carry the stage's scale words (TMA), which costs one stage of ring depth
  static constexpr int kStages = WT == 2 ? (TOK == 160 ? 4 : 3) : kFp4 ? (TOK <= 64 ? 3 : 2)
                                      : CPS == 2 ? (TOK <= 64 ? (MAXE <= 256 ? 4 : 3) : TOK <= 128 ? 3 : 2)
                                                 : TOK <= 64 ? 8 : TOK <= 224 ? 4 : 2;
  // NVFP4 scale words of one stage in shared memory: weights [4 MMAs][128 rows] int32 (box 128 x 4),
  // tokens [4 MMAs][TOK + 4] int32 (box TOK + 4 wide from the 4-aligned row at or below the tile's first)
  static constexpr int kSfTokCols = TOK + 4;
  static constexpr int kSfStageBytes = kFp4 ? 4 * kBlockW * 4 * WT + 4 * kSfTokCols * 4 : 0;
  static constexpr int kStageSf = (kSfStageBytes + 127) / 128 * 128;
  static constexpr int kAccBufs = kF32 ? 4 : (CPS == 1 && TOK <= 224 && WT == 1) ? 2 : 1;
  static constexpr int kTokSfCols = (TOK + 31) / 32;           // token-SF TMEM columns per MMA
  // NVFP4: token-SF columns of MMA k start every kTokSfStride columns (4-column aligned)
  static constexpr int kTokSfStride = kTokSfCols <= 4 ? 4 : 8;
  // NVFP4 with more than 128 tokens: two SF slots (2 x 192 accumulator columns + 2 x 64 = 512)
  static constexpr int kSfSlots = (kBf16 || kF32) ? 1 : kFp4 ? (TOK > 128 ? 2 : 4)
                                                             : (CPS == 1 && TOK <= 224 && WT == 1) ? 4 : 2;
  static_assert(kTokSfCols >= 1 && kTokSfCols <= 14, "token SF columns");
  static constexpr int kBoxRows = TOK <= 64 ? 32 : TOK <= 128 ? 64 : TOK == 160 ? 80 : TOK == 192 ? 64
                                 : TOK <= 224 ? 56 : 224;   // token rows per TMA box
  // Launched as a programmatic dependent of the preceding kernel (dispatch / route / quantise)
  // only for the small-batch tile: there the launch and prologue overlap that kernel's tail
  // (-0.9 us per graph-replayed decode step, -2 us eager).  The large-tile variants lost
  // 0.5-1 % as dependents in graph replay (same-box A/B), so they launch plainly.
  static constexpr bool kDependentLaunch = TOK <= 64;
  // The small-batch tile's work items all cost the same (one 128 x K weight tile streamed from
  // memory); run only as many CTAs as give every active CTA the same number of items.
  static constexpr bool kBalanceRounds = TOK <= 64;
  static constexpr int kSub = TOK <= 224 ? TOK : 224;         // MMA N of one sub-tile (<= 256)
  // SF slot: 4 weight-SF columns per weight tile, then per sub-tile kSub/32 token-SF columns
  // starting every 8 columns (scale-factor TMEM addresses stay 4-column aligned)
  static constexpr int kSubSfCols = kSub / 32;
  static constexpr int kWSfCols = 4 * WT;
  // NVFP4 slot: 16 weight-SF columns per weight tile (four MMAs x four), then four MMAs' token-SF
  // columns kTokSfStride apart
  static constexpr int kSfCols = (kBf16 || kF32) ? 0 : kFp4 ? 16 * WT + 4 * kTokSfStride
                                                          : TOK <= 64 ? 8 : TOK <= 224 ? 16 : 32;
  static __device__ __forceinline__ int tok_sf_col(int c) {
    return kWSfCols + (c / kSubSfCols) * 8 + c % kSubSfCols;
  }
  static constexpr int kAccCols = WT * TOK;                   // one accumulator: WT blocks of TOK columns
  static constexpr int kSfBase = kAccBufs * kAccCols;
  static constexpr int kTmemUsed = kSfBase + kSfSlots * kSfCols;
  static constexpr int kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                   : kTmemUsed <= 256 ? 256 : 512;
  static constexpr int kStageB = WT * kBlockW * kBlockK;      // bytes
  static constexpr int kStageA = TOK * kBlockK;
  // epilogue warps: one group of four (one per TMEM lane quadrant) per weight tile of the item, so
  // with WT = 2 both halves of the accumulator drain at once (the next item's MMAs wait for them)
  // FP32 scales with 128-token tiles: two groups of four epilogue warps each promote 64 of the
  // tile's token columns (64 FP32 accumulators per thread); the second group is warps 6-9, which
  // load no scale factors in this format
  static constexpr bool kF32Wide = kF32 && TOK == 128;
  static constexpr int kEpiGroups = (kF32Wide || WT == 2) ? 2 : 1;
  static constexpr int kEpiWarps = 4 * kEpiGroups;
  // warp 0 TMA producer, warp 1 MMA issuer, warps 2-5 epilogue group 0, warps 6-9 SF loaders
  // (epilogue group 1 when kF32Wide), warps 10.. further epilogue groups
  // WT = 2: one more warp, the waiter, performs every mbarrier wait of the MMA issuers and hands each
  // stage over through named barrier kHandoffBar, so no issuing thread reads shared memory; and a
  // second MMA-issuing warp (kIssuer2Warp) issues weight tile 1's MMAs while warp 1 issues tile 0's.
  // One issuing thread cannot keep the tensor core busy at N < ~176: each tcgen05.mma costs it ~70
  // cycles and each stage's hand-off ~100 more, against 72 cycles of tensor work per MMA at N = 144
  // (isolated issue loop, 8 MMAs per stage: one issuer 681 cycles per stage, two issuers 576 = the
  // tensor core's own time).
  static constexpr bool kWaiter = WT == 2;
  static constexpr int kWaiterWarp = 2 + kEpiWarps + 4;
  static constexpr int kIssuers = WT == 2 ? 2 : 1;
  static constexpr int kIssuer2Warp = kWaiterWarp + 1;
  static constexpr int kHandoffBar = 1;
  static constexpr int kHandoffThreads = 32 * (1 + kIssuers);   // waiter + issuing warps
  static constexpr int kNumThreads =
      kF32Wide ? 320 : 32 * (2 + kEpiWarps + 4 + (kWaiter ? 1 : 0) + (kIssuers - 1));
  // shared memory of the FP32-scale epilogue (per warp: the partial's column scales, and at the end of
  // a tile 32 tokens x 32 columns of bf16 for the transposed stores); the other epilogues store
  // straight from registers
  static constexpr int kEpiBytes = kF32 ? kEpiWarps * 32 * 32 * 2 : 0;
  static constexpr int kTableBytes = (3 * MAXE + 4) * 4;
  static constexpr int kBarBytes = 512;
  // full + empty per stage, sf_full + sf_empty per SF slot, acc_full + acc_empty per accumulator,
  // mma_done; then the TMEM base word and the abort flag
  static_assert((2 * kStages + 2 * kSfSlots + 2 * kAccBufs + 1) * 8 + 8 <= kBarBytes, "barrier region");
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * (kStageB + kStageA + kStageSf) +
                                  kEpiBytes + kTableBytes + kBarBytes;
  static_assert(kSfBase + kSfSlots * kSfCols <= 512, "TMEM columns");
  static_assert(kBf16 || kF32 || kWSfCols + (TOK / kSub - 1) * 8 + kSubSfCols <= kSfCols, "SF slot width");
  static_assert(WT == 1 || (WT == 2 && CPS == 1 && (((FMT == kFmtFp8 || FMT == kFmtBf16) && TOK == 224) ||
                                                    ((FMT == kFmtFp8 || FMT == kFmtBf16) && TOK == 160 && MAXE <= 256) ||
                                                    (FMT == kFmtNvfp4 && (TOK == 128 || TOK == 192)))),
                "two weight tiles per item, one CTA per SM: FP8 or BF16 with 224 tokens (or 160 tokens and at "
                "most 256 experts), NVFP4 with 128 or 192");
  static_assert(!kF32 || ((TOK == 64 || TOK == 128) && CPS == 1) || (TOK == 32 && CPS == 2),
                "FP32-scale tile: 64 or 128 tokens with one CTA per SM, or 32 with two (at most 64 FP32 "
                "accumulators per thread)");
  static_assert(kSubSfCols <= 8, "token SF columns of a sub-tile");
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static_assert(kSmem * CPS + 1024 * CPS <= 233472, "shared memory budget");
  static_assert(kTmemCols * CPS <= 512, "TMEM budget of the CTAs on one SM");
  static_assert(TOK % 32 == 0 && TOK <= 448, "token tile");
  static_assert(TOK % kBoxRows == 0, "whole TMA boxes must fit the token stage");
  static_assert(kSub % 32 == 0 && (kSub * kBlockK) % 1024 == 0, "sub-tile alignment");
  static_assert((kBoxRows * kBlockK) % 1024 == 0, "TMA boxes must keep the 1024-byte swizzle alignment");
  static_assert(!kFp4 || ((TOK <= 128 || (TOK == 192 && WT == 2)) && MAXE <= kNvfp4MaxE),
                "NVFP4 tiles: at most 128 tokens (192 in 256-row items), 256 experts");
};

struct Tile {
  int e, nt, tok0, ntok;
};

// 2**j for j clamped to [-100, 100] (exact).
__device__ __forceinline__ float exp2_int(int j) {
  j = j < -100 ? -100 : (j > 100 ? 100 : j);
  return __uint_as_float(static_cast<uint32_t>(127 + j) << 23);
}

__device__ __forceinline__ Tile decode_tile(int t, const int* tile_start, const int* row0, const int* cnt, int E,
                                            int nnt, int tok) {
  int lo = 0, hi = E - 1;   // last expert whose first tile is <= t (never an empty one)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int local = t - tile_start[lo];
  const int c = cnt[lo];
  const int nchunks = (c + tok - 1) / tok;
  const int nt = local / nchunks;
  const int chunk = local - nt * nchunks;
  // equal chunks (rounded up to 16 rows, never above tok): 264 rows -> 2 x 144
  const int per = min(tok, ((c + nchunks - 1) / nchunks + 15) & ~15);
  Tile r;
  r.e = lo;
  r.nt = nt;
  r.tok0 = row0[lo] + chunk * per;
  r.ntok = min(per, c - chunk * per);
  return r;
}

// acc[j] += partial[j] * scale[j] for 32 columns, two per packed FP32x2 FMA (each half rounded once,
// as fmaf); the scales come from shared memory as float4 broadcasts.
__device__ __forceinline__ void promote32(float* acc, const uint32_t (&r)[32], const float* scale) {
#pragma unroll
  for (int j4 = 0; j4 < 8; ++j4) {
    const float4 s4 = reinterpret_cast<const float4*>(scale)[j4];
    fma2_f32(acc[4 * j4], acc[4 * j4 + 1], __uint_as_float(r[4 * j4]), __uint_as_float(r[4 * j4 + 1]), s4.x, s4.y);
    fma2_f32(acc[4 * j4 + 2], acc[4 * j4 + 3], __uint_as_float(r[4 * j4 + 2]), __uint_as_float(r[4 * j4 + 3]), s4.z,
             s4.w);
  }
}

// Bounded wait that ignores the abort flag (used while draining at exit).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Wait in every lane of a warp; the warp proceeds only if all lanes saw the
// phase complete, so the .sync.aligned tcgen05 ops that follow stay uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
  const bool ok = mbar_wait(bar, parity, abort, err);
  return __all_sync(0xffffffffu, ok);
}

template <int TOK, int CPS, int MAXE, int FMT, int WT>
__global__ void __launch_bounds__(Cfg<TOK, CPS, MAXE, FMT, WT>::kNumThreads, CPS)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_sfb, const __grid_constant__ CUtensorMap tmap_sfa,
                        const GemmArgs p) {
  using C = Cfg<TOK, CPS, MAXE, FMT, WT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_b = smem;
  uint8_t* stage_a = stage_b + C::kStages * C::kStageB;
  uint8_t* stage_sf = stage_a + C::kStages * C::kStageA;    // NVFP4 only (kStageSf = 0 otherwise)
  uint8_t* epi = stage_sf + C::kStages * C::kStageSf;
  int* tile_start = reinterpret_cast<int*>(epi + C::kEpiBytes);
  int* exp_row0 = tile_start + C::kMaxE + 1;
  int* exp_cnt = exp_row0 + C::kMaxE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(tile_start) + C::kTableBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + C::kStages;
  uint64_t* sf_full = empty + C::kStages;
  uint64_t* sf_empty = sf_full + C::kSfSlots;
  uint64_t* acc_full = sf_empty + C::kSfSlots;
  uint64_t* acc_empty = acc_full + C::kAccBufs;
  uint64_t* mma_done = acc_empty + C::kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E, N = p.N;
  const int nnt = N / kBlockW;                               // 128-row weight tiles per expert
  const int nit = nnt / WT;                                  // work-item columns per token chunk
  const int nkb = p.K / C::kKElems;
  const int nw = C::kFp4 ? p.K / 64 : (nkb + 3) / 4;        // SF words per row

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], (C::kFp4 ? 4 : 0) + C::kIssuers);   // the MMA commits (+ NVFP4: the four SF warps)
    }
    for (int s = 0; s < C::kSfSlots; ++s) {
      mbar_init(&sf_full[s], 4);
      mbar_init(&sf_empty[s], C::kIssuers);
    }
    for (int s = 0; s < C::kAccBufs; ++s) {
      mbar_init(&acc_full[s], C::kIssuers);
      mbar_init(&acc_empty[s], C::kEpiWarps);
    }
    mbar_init(mma_done, C::kIssuers);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_a);
    if (C::kFp4) {
      tma_prefetch_desc(&tmap_sfb);
      tma_prefetch_desc(&tmap_sfa);
    }
  }
  // Dependent launch: the weights are not written by the preceding kernel, so while it drains,
  // start pulling into L2 the first stages of the tile this CTA most likely takes first (tile
  // blockIdx.x when every expert holds one token chunk, as at decode).  A wrong guess costs only
  // bandwidth.  Weights in host memory are left alone (every byte crosses the host link).
  if (C::kDependentLaunch && warp == 0 && lane == 0 && !(p.flags & BSF_B_HOST_MAPPED)) {
    const int e = static_cast<int>(blockIdx.x) / nnt, nt = static_cast<int>(blockIdx.x) % nnt;
    if (e < E) {
      const int n_pf = nkb < kPrefetchStages ? nkb : kPrefetchStages;
      for (int kb = 0; kb < n_pf; ++kb) {
        if (p.flags & BSF_B_TILED)
          tma_prefetch_l2(&tmap_b, 0, ((e * nnt + nt) * nkb + kb) * kBlockW);
        else
          tma_prefetch_l2(&tmap_b, kb * kBlockK, e * N + nt * kBlockW);
      }
    }
  }
  // when launched as a dependent, everything above overlaps the tail of the preceding kernel;
  // nothing the preceding kernel writes, and no tensor memory, is touched before it has completed
  // (no-op otherwise)
  pdl_wait();
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2) {
    // per-expert rows and tile offsets (exclusive scan over experts, 32 at a time)
    int carry = 0;
    int bad = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int row0 = 0, cnt = 0;
      if (e < E) {
        cnt = p.counts[e];
        if (p.seg_start == nullptr) {
          row0 = static_cast<int>(e * p.max_m);
          if (cnt < 0 || cnt > p.max_m) { bad = 1; cnt = cnt < 0 ? 0 : static_cast<int>(p.max_m); }
        } else {
          row0 = p.seg_start[e];
          if (cnt < 0 || row0 < 0 || static_cast<int64_t>(row0) + cnt > p.m_rows) { bad = 1; cnt = 0; }
        }
        exp_row0[e] = row0;
        exp_cnt[e] = cnt;
      }
      const int ntiles = ((cnt + TOK - 1) / TOK) * nit;
      int incl = ntiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) tile_start[e] = carry + incl - ntiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tile_start[E] = carry;
    if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0) raise_error(p.err, BSF_DEVERR_SEGMENT);
  }
  __syncwarp();   // warp 0 reconverges after the single-lane set-up before the block barrier
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_start[E];
  // CTA b takes tiles b, b + G, b + 2G, ...  With equal-cost tiles, G is lowered to the fewest
  // CTAs that still need no more rounds than the whole grid would (3072 tiles on 304 CTAs:
  // 280 CTAs x 11 instead of 32 CTAs running an 11th tile alone, pipeline-limited).
  int G = static_cast<int>(gridDim.x);
  if (C::kBalanceRounds && total_tiles > 0) {
    const int rounds = (total_tiles + G - 1) / G;
    G = (total_tiles + rounds - 1) / rounds;
  }
  const int t_first = static_cast<int>(blockIdx.x) < G ? static_cast<int>(blockIdx.x) : total_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = !(p.flags & BSF_DEBUG_WITHHOLD_LOADS);
      for (int t = t_first; t < total_tiles && ok; t += G) {
        const Tile tl = decode_tile(t, tile_start, exp_row0, exp_cnt, E, nit, TOK);
        const int n_loads = (tl.ntok + C::kBoxRows - 1) / C::kBoxRows;
        const uint32_t bytes = C::kStageB + n_loads * C::kBoxRows * kBlockK + C::kSfStageBytes;
        const int wt0 = tl.nt * WT;                          // first 128-row weight tile of the item
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
          for (int w = 0; w < WT; ++w) {
            uint8_t* dst = stage_b + stage * C::kStageB + w * kBlockW * kBlockK;
            if (p.flags & BSF_B_TILED)   // weights pre-tiled: box (e, weight tile, kb) is 16 KB contiguous
              tma_load_2d(dst, &tmap_b, &full[stage], 0, ((tl.e * nnt + wt0 + w) * nkb + kb) * kBlockW);
            else
              tma_load_2d(dst, &tmap_b, &full[stage], kb * kBlockK, tl.e * N + (wt0 + w) * kBlockW);
          }
          for (int i = 0; i < n_loads; ++i)
            tma_load_2d(stage_a + stage * C::kStageA + i * C::kBoxRows * kBlockK, &tmap_a, &full[stage],
                        kb * kBlockK, tl.tok0 + i * C::kBoxRows);
          if (C::kFp4) {
            // scale words of MMAs 4kb .. 4kb+3: weight rows of the tile, and the tile's token rows
            // from the 4-aligned row at or below tok0 (the x coordinate of a TMA copy must be 16-byte aligned)
            uint8_t* sf_dst = stage_sf + stage * C::kStageSf;
#pragma unroll
            for (int w = 0; w < WT; ++w)
              tma_load_2d(sf_dst + w * 4 * kBlockW * 4, &tmap_sfb, &full[stage], (tl.nt * WT + w) * kBlockW,
                          tl.e * nw + kb * 4);
            tma_load_2d(sf_dst + WT * 4 * kBlockW * 4, &tmap_sfa, &full[stage], tl.tok0 & ~3, kb * 4);
          }
          ++issued;
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // make sure no TMA write is still in flight when the CTA exits
      const int outstanding = issued < C::kStages ? issued : C::kStages;
      for (int j = 0; j < outstanding; ++j) {
        if (stage == 0) { stage = C::kStages; phase ^= 1u; }
        --stage;
        drain_wait(&full[stage], phase);
      }
    }
  } else if (warp == 1 || (C::kIssuers == 2 && warp == C::kIssuer2Warp)) {
    // ------------------------------------------------------------ MMA issuer(s)
    if (C::kF32 && lane == 0) {
      // one partial accumulator per 128-K stage, alternating between the two TMEM buffers
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = t_first; t < total_tiles && ok; t += G) {
        const Tile tl = decode_tile(t, tile_start, exp_row0, exp_cnt, E, nit, TOK);
        const uint32_t mma_n = (tl.ntok + 15) & ~15;
        const uint32_t idesc = idesc_f8(kBlockW, mma_n);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.err)) { ok = false; break; }
          if (!mbar_wait(&full[stage], phase, abort_flag, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t adesc = smem_desc_k_sw128(smem_u32(stage_b + stage * C::kStageB));
          const uint64_t bdesc = smem_desc_k_sw128(smem_u32(stage_a + stage * C::kStageA));
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_f8(tmem_base + acc * TOK, adesc + 2 * k, bdesc + 2 * k, idesc, k != 0);
          tc_commit(&empty[stage]);
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
          tc_commit(&acc_full[acc]);
          if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
        }
      }
      tc_commit(mma_done);
      drain_wait(mma_done, 0);
    } else if (!C::kF32) {
      // One stage's MMAs (K = 128 bytes of both operands) into accumulator d_tmem, issued as
      // straight-line code: a branch between two tcgen05.mma instructions stalls the tensor pipe.
      // With two issuers, each issues the MMAs of its own weight tile w_first (kWN = 1).  The two-tile
      // items issue in the warp-wide form (every lane runs this code, lane 0 issues).
      constexpr int kWN = C::kIssuers == 2 ? 1 : WT;
      const int w_first = warp == 1 ? 0 : 1;
      const uint32_t lead = lane == 0;
      auto issue_stage = [&](uint32_t stage, uint32_t sf_slot, uint32_t d_tmem, uint32_t mma_n, int kb) {
        const uint32_t sfw = tmem_base + C::kSfBase + sf_slot * C::kSfCols;
        const uint32_t sft = sfw + C::kWSfCols;
        const uint64_t adesc = smem_desc_k_sw128(smem_u32(stage_b + stage * C::kStageB));
        const uint64_t bdesc = smem_desc_k_sw128(smem_u32(stage_a + stage * C::kStageA));
        if constexpr (C::kFp4) {
          // four K = 64 steps; step k's scales: weight words at columns 4k, token words at 16 + 4k
          // (NVFP4 tiles hold at most 192 tokens: one sub-tile, MMA N = mma_n <= 192)
          static_assert(!C::kFp4 || TOK == C::kSub, "NVFP4: one MMA sub-tile");
          // (two weight tiles: tile w's words at 16 w + 4k, token words at 16 WT + 4k)
          const uint32_t idesc = idesc_nvf4(kBlockW, mma_n);
          uint64_t adw[kWN];
#pragma unroll
          for (int ww = 0; ww < kWN; ++ww)
            adw[ww] = smem_desc_k_sw128(smem_u32(stage_b + stage * C::kStageB + (w_first + ww) * kBlockW * kBlockK));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int ww = 0; ww < kWN; ++ww) {
              const int w = w_first + ww;
              if constexpr (C::kWaiter)
                mma_nvf4_if(d_tmem + w * TOK, adw[ww] + 2 * k, bdesc + 2 * k, idesc, sfw + 16 * w + 4 * k,
                            sfw + 16 * WT + C::kTokSfStride * k, (kb | k) != 0, lead);
              else
                mma_nvf4(d_tmem + w * TOK, adw[ww] + 2 * k, bdesc + 2 * k, idesc, sfw + 16 * w + 4 * k,
                         sfw + 16 * WT + C::kTokSfStride * k, (kb | k) != 0);
            }
          }
        } else {
        // sub-tiles of at most kSub tokens: columns j*kSub.., smem rows j*kSub.., token SF columns j*kSub/32..
#pragma unroll
        for (int j = 0; j < TOK / C::kSub; ++j) {
          const int n_j = static_cast<int>(mma_n) - j * C::kSub;
          if (n_j <= 0) break;
          const uint32_t nn = n_j < C::kSub ? n_j : C::kSub;    // MMA N of this sub-tile: 16..224
          const uint64_t bd = bdesc + static_cast<uint64_t>(j * C::kSub * kBlockK >> 4);
          if constexpr (C::kBf16) {
            // four K = 16 steps of 32 bytes inside the swizzled 128-byte rows
            const uint32_t idesc = idesc_bf16(kBlockW, nn);
            uint64_t adw[kWN];
#pragma unroll
            for (int ww = 0; ww < kWN; ++ww)
              adw[ww] = smem_desc_k_sw128(smem_u32(stage_b + stage * C::kStageB + (w_first + ww) * kBlockW * kBlockK));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
              for (int ww = 0; ww < kWN; ++ww) {
                const int w = w_first + ww;
                if constexpr (C::kWaiter)
                  mma_bf16_if(d_tmem + w * TOK + j * C::kSub, adw[ww] + 2 * k, bd + 2 * k, idesc, (kb | k) != 0, lead);
                else
                  mma_bf16(d_tmem + w * TOK + j * C::kSub, adw[ww] + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
              }
            }
          } else {
            const uint32_t idesc = idesc_mxf8_e4m3(kBlockW, nn, kb & 3, kb & 3);
            uint64_t adw[kWN];             // weight tile w of the stage; its accumulator block and SF columns
#pragma unroll
            for (int ww = 0; ww < kWN; ++ww)
              adw[ww] = smem_desc_k_sw128(smem_u32(stage_b + stage * C::kStageB + (w_first + ww) * kBlockW * kBlockK));
#pragma unroll
            for (int k = 0; k < kBlockK / 32; ++k) {
              // advance 32 bytes (one K=32 step of FP8) inside the swizzled 128-byte rows
#pragma unroll
              for (int ww = 0; ww < kWN; ++ww) {
                const int w = w_first + ww;
                if constexpr (C::kWaiter)
                  mma_mxf8_if(d_tmem + w * TOK + j * C::kSub, adw[ww] + 2 * k, bd + 2 * k, idesc, sfw + 4 * w,
                              sft + j * 8, (kb | k) != 0, lead);
                else
                  mma_mxf8(d_tmem + w * TOK + j * C::kSub, adw[ww] + 2 * k, bd + 2 * k, idesc, sfw + 4 * w,
                           sft + j * 8, (kb | k) != 0);
              }
            }
          }
        }
        }
      };
      if constexpr (C::kWaiter) {
        // The issuing threads read no shared memory between stages: any load there (an mbarrier
        // wait, even on a completed phase, or a plain flag) lets the tensor pipe drain before the
        // next MMAs (measured: a 4-MMA stage of N = 128 grows from 256 to ~440 cycles).  The waiter
        // warp does every wait and hands each stage over through named barrier kHandoffBar, whose
        // OR-reduced predicate carries an abort.  Each issuing warp runs the loop whole; its lane 0
        // issues its weight tile's MMAs and commits, so every barrier the MMAs release counts one
        // arrival per issuer.
        uint32_t stage = 0, sf_slot = 0, acc = 0;
        bool ok = true;
        for (int t = t_first; t < total_tiles && ok; t += G) {
          const Tile tl = decode_tile(t, tile_start, exp_row0, exp_cnt, E, nit, TOK);
          const uint32_t mma_n = (tl.ntok + 15) & ~15;
          const uint32_t d_tmem = tmem_base + acc * C::kAccCols;
          for (int kb = 0; kb < nkb; ++kb) {
            // this stage's data (for kb = 0 also the drained accumulator; per slot the scales) is ready
            if (named_barrier_or(C::kHandoffBar, C::kHandoffThreads, false)) { ok = false; break; }
            tc_fence_after();
            issue_stage(stage, sf_slot, d_tmem, mma_n, kb);
            tc_commit_if(&empty[stage], lead);
            const bool slot_done = !C::kBf16 && (kb % C::kKbPerSlot == C::kKbPerSlot - 1 || kb == nkb - 1);
            if (slot_done) tc_commit_if(&sf_empty[sf_slot], lead);
            if (++stage == C::kStages) stage = 0;
            if (slot_done && ++sf_slot == C::kSfSlots) sf_slot = 0;
          }
          if (!ok) break;
          tc_commit_if(&acc_full[acc], lead);
          if (++acc == C::kAccBufs) acc = 0;
        }
        // wait for every MMA issued by this warp's lane 0 (and, through the barrier's count, by the
        // other issuer) before TMEM can be released
        tc_commit_if(mma_done, lead);
        if (lane == 0) drain_wait(mma_done, 0);
      } else if (lane == 0) {
      uint32_t stage = 0, phase = 0, sf_slot = 0, sf_phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = t_first; t < total_tiles && ok; t += G) {
        const Tile tl = decode_tile(t, tile_start, exp_row0, exp_cnt, E, nit, TOK);
        const uint32_t mma_n = (tl.ntok + 15) & ~15;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::kAccCols;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!C::kBf16 && kb % C::kKbPerSlot == 0) {
            if (!mbar_wait(&sf_full[sf_slot], sf_phase, abort_flag, p.err)) { ok = false; break; }
          }
          if (!mbar_wait(&full[stage], phase, abort_flag, p.err)) { ok = false; break; }
          tc_fence_after();
          issue_stage(stage, sf_slot, d_tmem, mma_n, kb);
          tc_commit(&empty[stage]);
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
          if (!C::kBf16 && (kb % C::kKbPerSlot == C::kKbPerSlot - 1 || kb == nkb - 1)) {
            tc_commit(&sf_empty[sf_slot]);
            if (++sf_slot == C::kSfSlots) { sf_slot = 0; sf_phase ^= 1u; }
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
      }
      // wait for every MMA issued by this thread before TMEM can be released
      tc_commit(mma_done);
      drain_wait(mma_done, 0);
      }
    }
    __syncwarp();
  } else if (C::kWaiter && warp == C::kWaiterWarp) {
    // ------------------------------------------------------------ waiter (two-weight-tile items)
    // Every wait of the MMA issuer, in the issuer's order; each stage is handed over through the
    // named barrier (the OR of its predicate tells the issuer to stop).
    uint32_t stage = 0, phase = 0, sf_slot = 0, sf_phase = 0, acc = 0, acc_phase = 0;
    bool ok = true;
    for (int t = t_first; t < total_tiles && ok; t += G) {
      for (int kb = 0; kb < nkb; ++kb) {
        bool good = kb != 0 || warp_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.err);
        if (good && !C::kBf16 && kb % C::kKbPerSlot == 0) good = warp_wait(&sf_full[sf_slot], sf_phase, abort_flag, p.err);
        if (good) good = warp_wait(&full[stage], phase, abort_flag, p.err);
        if (named_barrier_or(C::kHandoffBar, C::kHandoffThreads, !good)) { ok = false; break; }
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        if (!C::kBf16 && (kb % C::kKbPerSlot == C::kKbPerSlot - 1 || kb == nkb - 1))
          if (++sf_slot == C::kSfSlots) { sf_slot = 0; sf_phase ^= 1u; }
      }
      if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
    }
  } else if (warp < 6 || (warp >= 10 && warp < 10 + 4 * (C::kEpiGroups - 1)) || (C::kF32Wide && warp < 10)) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quadrant = weight rows 32q..32q+31
    const int ew = warp < 10 ? warp - 2 : warp - 6;  // epilogue warp 0 .. kEpiWarps-1
    const int group = ew / 4;                          // handles weight tiles group, group + kEpiGroups, ...
    uint16_t* buf = reinterpret_cast<uint16_t*>(epi) + ew * 32 * 32;   // FP32-scale epilogue only
    uint32_t acc = 0, acc_phase = 0;
    if constexpr (C::kF32) {
      // D[token, row] = sum_kb sB[e, nt, kb] * sA[token, kb] * partial_kb: promoted in FP32 registers,
      // in K-block order; lane = weight row 32q + lane, accv[j] = token j of the tile
      const int nnb = N / kBlockW;
      bool ok = true;
      for (int t = t_first; t < total_tiles && ok; t += G) {
        const Tile tl = decode_tile(t, tile_start, exp_row0, exp_cnt, E, nit, TOK);
        // this warp group's token columns gt0 .. gt0 + kGT - 1 of the tile
        constexpr int kGT = TOK / C::kEpiGroups;
        // the 128-token tile (large batches) reads the column scales from shared memory as float4
        // broadcasts and uses packed FP32x2 FMAs; the small tiles (register-capped, HBM-bound) keep
        // the per-column shuffle
        constexpr bool kSmemScales = TOK == 128;
        const int gt0 = group * kGT;
        float accv[kGT];
#pragma unroll
        for (int j = 0; j < kGT; ++j) accv[j] = 0.f;
        const float* sbp = p.sfb_f32 + (static_cast<int64_t>(tl.e) * nnb + tl.nt) * nkb;
        const int64_t r0 = static_cast<int64_t>(tl.tok0) + gt0 + lane;
        // the scales of K-blocks kb .. kb+3 are in flight ahead of their partials.  The 128-token tile
        // keeps them in a ring of four register slots, K-block kb in slot kb % 4, with the K-block loop
        // unrolled by four: a slot is refilled right after it is read and not read again for four
        // K-blocks.  (A shifting queue makes every K-block wait for the loads issued one K-block
        // earlier: large gate-up 3.59 ms with it.)
        float qb[4], q0[4], q1[4];
        auto fetch = [&](int kk, float& b, float& s0, float& s1) {
          b = s0 = s1 = 0.f;
          if (kk < nkb) {
            const float* sap = p.sfa_f32 + static_cast<int64_t>(kk) * p.sfa_ld;
            b = __ldg(sbp + kk);
            if (gt0 + lane < tl.ntok) s0 = __ldg(sap + r0);
            if (gt0 + lane + 32 < tl.ntok) s1 = __ldg(sap + r0 + 32);
          }
        };
#pragma unroll
        for (int i = 0; i < 4; ++i) fetch(i, qb[i], q0[i], q1[i]);
        // one K-block: its partial scaled by sB * sA[token] and added into accv; false if a wait gave up
        auto kblock = [&](const float sb, const float sa0, const float sa1) -> bool {
          // column j's scale sB * sA[token j] is the same for every row (lane): lane j computes it once
          // into the warp's scratch, and every lane reads it back as a float4 broadcast
          float* sc = reinterpret_cast<float*>(buf);
          if constexpr (kSmemScales) {
            sc[lane] = sb * sa0;
            if constexpr (kGT > 32) sc[32 + lane] = sb * sa1;
            __syncwarp();
          }
          if (!warp_wait(&acc_full[acc], acc_phase, abort_flag, p.err)) return false;
          tc_fence_after();
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * TOK + gt0;
          uint32_t r[32];
          if (gt0 < tl.ntok) {
            tmem_ld_x32(taddr, r);
            tmem_wait_ld_regs(r);
            if constexpr (kSmemScales) {
              promote32(accv, r, sc);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                accv[j] = fmaf(__uint_as_float(r[j]), sb * __shfl_sync(0xffffffffu, sa0, j), accv[j]);
            }
          }
          if constexpr (kGT > 32) {
          if (tl.ntok > gt0 + 32) {
            tmem_ld_x32(taddr + 32, r);
            tmem_wait_ld_regs(r);
            if constexpr (kSmemScales) {
              promote32(accv + 32, r, sc + 32);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                accv[32 + j] = fmaf(__uint_as_float(r[j]), sb * __shfl_sync(0xffffffffu, sa1, j), accv[32 + j]);
            }
          }
          }
          tc_fence_before();
          __syncwarp();         // (the scratch is rewritten next stage)
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
          if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
          return true;
        };
        if constexpr (kSmemScales) {
          for (int kb0 = 0; kb0 < nkb && ok; kb0 += 4) {
#pragma unroll
            for (int slot = 0; slot < 4; ++slot) {
              const int kb = kb0 + slot;
              if (kb >= nkb) break;
              const float sb = qb[slot], sa0 = q0[slot], sa1 = q1[slot];
              fetch(kb + 4, qb[slot], q0[slot], q1[slot]);
              if (!kblock(sb, sa0, sa1)) { ok = false; break; }
            }
          }
        } else {
          // the small tiles (register-capped) keep a shifting queue
          for (int kb = 0; kb < nkb; ++kb) {
            const float sb = qb[0], sa0 = q0[0], sa1 = q1[0];
#pragma unroll
            for (int i = 0; i < 3; ++i) {
              qb[i] = qb[i + 1];
              q0[i] = q0[i + 1];
              q1[i] = q1[i + 1];
            }
            fetch(kb + 4, qb[3], q0[3], q1[3]);
            if (!kblock(sb, sa0, sa1)) { ok = false; break; }
          }
        }
        if (!ok) break;
#pragma unroll
        for (int half = 0; half < kGT / 32; ++half) {
          const int c0 = gt0 + 32 * half;             // token column of the tile
          if (c0 >= tl.ntok) break;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const __nv_bfloat16 h = __float2bfloat16_rn(accv[32 * half + j]);
            buf[j * 32 + lane] = *reinterpret_cast<const uint16_t*>(&h);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = (lane >> 2) + 8 * i;
            if (c0 + j < tl.ntok) {
              const uint4 v = *reinterpret_cast<const uint4*>(buf + j * 32 + (lane & 3) * 8);
              uint16_t* dst = p.d + static_cast<int64_t>(tl.tok0 + c0 + j) * N + tl.nt * kBlockW + 32 * q +
                              (lane & 3) * 8;
              *reinterpret_cast<uint4*>(dst) = v;
            }
          }
          __syncwarp();
        }
      }
    } else
    for (int t = t_first; t < total_tiles; t += G) {
      const Tile tl = decode_tile(t, tile_start, exp_row0, exp_cnt, E, nit, TOK);
      if (!warp_wait(&acc_full[acc], acc_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * C::kAccCols;
      const int ncol = (tl.ntok + 31) & ~31;
      // NVFP4: the tensor scales 2**a_exp * 2**b_exp[e], applied exactly (two power-of-two products)
      float alpha_a = 1.f, alpha_b = 1.f;
      if constexpr (C::kFp4) {
        alpha_a = exp2_int(p.a_exp);
        alpha_b = exp2_int(p.b_exp ? p.b_exp[tl.e] : 0);
      }
      // weight tile w of the item: accumulator columns w * TOK.., output columns (nt * WT + w) * 128..
      for (int w = group; w < WT; w += C::kEpiGroups) {
      const uint32_t taddr = tacc + w * TOK;
      // chunk c0's 32 token columns -> bf16, stored straight from registers: lane l holds weight row
      // 32q + l of every token; after one exchange with the neighbour lane, even lanes hold rows
      // (l, l + 1) of token j and odd lanes rows (l - 1, l) of token j + 1, so each store writes 4
      // bytes and a warp's store covers two tokens' 64-byte row segments.  (The earlier shared-memory
      // transpose, 2-byte stores into a buffer then 16-byte loads and stores, cost 3-4 % of the
      // large-M GEMMs: same-box A/B, bit-identical outputs.)
      auto emit = [&](const uint32_t (&r)[32], int c0) {
        const int odd = lane & 1;
        uint16_t* dst = p.d + static_cast<int64_t>(tl.tok0 + c0 + odd) * N +
                        static_cast<int64_t>(tl.nt * WT + w) * kBlockW + 32 * q + (lane & ~1);
#pragma unroll
        for (int jj = 0; jj < 32; jj += 2) {
          float v0 = __uint_as_float(r[jj]), v1 = __uint_as_float(r[jj + 1]);
          if constexpr (C::kFp4) {
            v0 = v0 * alpha_a * alpha_b;
            v1 = v1 * alpha_a * alpha_b;
          }
          const float x = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
          const uint32_t pk = odd ? pack_bf16x2(x, v1) : pack_bf16x2(v0, x);
          if (c0 + jj + odd < tl.ntok) *reinterpret_cast<uint32_t*>(dst + static_cast<int64_t>(jj) * N) = pk;
        }
      };
      // last chunk of the item in registers: hand the accumulator back to the MMA issuers
      auto release_if_last = [&](int c0) {
        if (w + C::kEpiGroups >= WT && c0 + 32 >= ncol) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
      };
      for (int c0 = 0; c0 < ncol; c0 += 32) {
        uint32_t r[32];
        tmem_ld_x32(taddr + c0, r);
        tmem_wait_ld_regs(r);
        release_if_last(c0);
        emit(r, c0);
      }
      }
      if (ncol == 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
      }
      if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
    }
  } else {
    // ------------------------------------------------------------ scale-factor loaders
    // Each of the four warps writes the same SF words into its own TMEM lane
    // quadrant: column c of a block holds rows (lane + 32 c), byte j = K-block 4g + j.
    const int q = warp & 3;
    uint32_t sf_slot = 0, sf_phase = 0;
    bool ok = true;
    if constexpr (C::kBf16 || C::kF32) {
      // no scale factors in tensor memory
    } else if constexpr (C::kFp4) {
      // NVFP4: the stage's scale words arrive with its data (TMA into shared memory); per stage,
      // MMA k's word of weight row (lane + 32c) of weight tile w -> TMEM column 16w + 4k + c, of token
      // row (lane + 32c) -> column 16 WT + kTokSfStride k + c (rows past the tile: scale 0).  The shared-memory stage is released
      // (one of the five arrivals on its empty barrier) as soon as the words are in registers.
      uint32_t stage = 0, phase = 0;
      for (int t = t_first; t < total_tiles && ok; t += G) {
        const Tile tl = decode_tile(t, tile_start, exp_row0, exp_cnt, E, nit, TOK);
        const int off = tl.tok0 & 3;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!warp_wait(&full[stage], phase, abort_flag, p.err)) { ok = false; break; }
          const uint32_t* sw = reinterpret_cast<const uint32_t*>(stage_sf + stage * C::kStageSf);
          const uint32_t* st = sw + 4 * kBlockW * WT;
          uint32_t w[WT][4][4];            // weight tile ww, MMA k, rows lane + 32 c
          uint32_t a[4][C::kTokSfCols];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int ww = 0; ww < WT; ++ww) {
#pragma unroll
              for (int c = 0; c < 4; ++c) w[ww][k][c] = sw[(ww * 4 + k) * kBlockW + 32 * c + lane];
            }
#pragma unroll
            for (int c = 0; c < C::kTokSfCols; ++c) {
              const int rl = lane + 32 * c;
              a[k][c] = rl < tl.ntok ? st[k * C::kSfTokCols + off + rl] : 0u;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
          if (!warp_wait(&sf_empty[sf_slot], sf_phase ^ 1u, abort_flag, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t col =
              tmem_base + (static_cast<uint32_t>(32 * q) << 16) + C::kSfBase + sf_slot * C::kSfCols;
#pragma unroll
          for (int ww = 0; ww < WT; ++ww) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tmem_st_x4(col + 16 * ww + 4 * k, w[ww][k][0], w[ww][k][1], w[ww][k][2], w[ww][k][3]);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int c = 0; c < C::kTokSfCols; ++c) tmem_st_x1(col + 16 * WT + C::kTokSfStride * k + c, a[k][c]);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sf_full[sf_slot]);
          if (++sf_slot == C::kSfSlots) { sf_slot = 0; sf_phase ^= 1u; }
        }
      }
    } else
    for (int t = t_first; t < total_tiles && ok; t += G) {
      const Tile tl = decode_tile(t, tile_start, exp_row0, exp_cnt, E, nit, TOK);
      const int mma_n = (tl.ntok + 15) & ~15;
      const int32_t* sfb_base = p.sfb + static_cast<int64_t>(tl.e) * nw * N + tl.nt * WT * kBlockW + lane;
      for (int g = 0; g < nw; ++g) {
        uint32_t w[WT][4];             // weight tile w: rows lane + 32 c of the item's tile w
#pragma unroll
        for (int ww = 0; ww < WT; ++ww) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            w[ww][c] = static_cast<uint32_t>(__ldg(sfb_base + static_cast<int64_t>(g) * N + ww * kBlockW + 32 * c));
        }
        uint32_t a[C::kTokSfCols];
#pragma unroll
        for (int c = 0; c < C::kTokSfCols; ++c) {
          const int rl = lane + 32 * c;
          const int64_t row = static_cast<int64_t>(tl.tok0) + rl;
          a[c] = (rl < mma_n && row < p.m_rows) ? static_cast<uint32_t>(__ldg(p.sfa + g * p.sfa_ld + row))
                                                 : 0x7F7F7F7Fu;
        }
        if (!warp_wait(&sf_empty[sf_slot], sf_phase ^ 1u, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t col = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + C::kSfBase + sf_slot * C::kSfCols;
#pragma unroll
        for (int ww = 0; ww < WT; ++ww) tmem_st_x4(col + 4 * ww, w[ww][0], w[ww][1], w[ww][2], w[ww][3]);
#pragma unroll
        for (int c = 0; c < C::kTokSfCols; ++c) tmem_st_x1(col + C::tok_sf_col(c), a[c]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_full[sf_slot]);
        if (++sf_slot == C::kSfSlots) { sf_slot = 0; sf_phase ^= 1u; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
template <int TOK, int CPS = 1, int MAXE = kMaxExperts, int FMT = kFmtFp8, int WT = 1>
bsf_status launch(const GemmArgs& args, const uint8_t* a, const uint8_t* b, int64_t max_tiles, cudaStream_t s) {
  using C = Cfg<TOK, CPS, MAXE, FMT, WT>;
  if (args.E > MAXE) return BSF_ERR_UNSUPPORTED;
  CUtensorMap map_a, map_b;
  const int64_t row_bytes = C::kFp4 ? args.K / 2 : C::kBf16 ? 2 * args.K : args.K;
  if (!make_map(&map_a, a, args.m_rows, row_bytes, C::kBoxRows)) return BSF_ERR_CUDA;
  if (args.flags & BSF_B_TILED) {   // [E][N/128][row_bytes/128] boxes of 128 rows x 128 bytes, each contiguous
    if (static_cast<int64_t>(args.E) * args.N * (row_bytes / 128) > INT32_MAX) return BSF_ERR_UNSUPPORTED;
    if (!make_map(&map_b, b, static_cast<int64_t>(args.E) * args.N * (row_bytes / 128), 128, kBlockW))
      return BSF_ERR_CUDA;
  } else if (!make_map(&map_b, b, static_cast<int64_t>(args.E) * args.N, row_bytes, kBlockW)) {
    return BSF_ERR_CUDA;
  }
  CUtensorMap map_sfb = map_b, map_sfa = map_a;     // placeholders: only NVFP4 stages load scale words by TMA
  if (C::kFp4) {
    const int64_t nw = args.K / 64;
    if (!make_map_i32(&map_sfb, args.sfb, static_cast<int64_t>(args.E) * nw, args.N, kBlockW, 4)) return BSF_ERR_CUDA;
    if (!make_map_i32(&map_sfa, args.sfa, nw, args.sfa_ld, C::kSfTokCols, 4)) return BSF_ERR_CUDA;
  }
  static std::atomic<bool> attr_set[64];   // setting the attributes twice (racing first calls) is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(grouped_gemm_kernel<TOK, CPS, MAXE, FMT, WT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::kSmem)) != cudaSuccess)
      return BSF_ERR_CUDA;
    if (CPS > 1 && cudaFuncSetAttribute(grouped_gemm_kernel<TOK, CPS, MAXE, FMT, WT>,
                                        cudaFuncAttributePreferredSharedMemoryCarveout,
                                        cudaSharedmemCarveoutMaxShared) != cudaSuccess)
      return BSF_ERR_CUDA;
    attr_set[dev].store(true, std::memory_order_release);
  }
  int64_t grid = static_cast<int64_t>(sm_count()) * CPS;
  if (max_tiles < grid) grid = max_tiles;
  if (grid <= 0) return BSF_OK;
  if (C::kDependentLaunch)
    return launch_dependent(grouped_gemm_kernel<TOK, CPS, MAXE, FMT, WT>, static_cast<unsigned>(grid), C::kNumThreads, C::kSmem, s,
                            map_b, map_a, map_sfb, map_sfa, args);
  grouped_gemm_kernel<TOK, CPS, MAXE, FMT, WT><<<static_cast<unsigned>(grid), C::kNumThreads, C::kSmem, s>>>(
      map_b, map_a, map_sfb, map_sfa, args);
  return launch_status();
}

// With BSF_B_HOST_MAPPED, b and sfb are pinned host allocations; the kernel
// reads them through their device-mapped addresses ("AsymGEMM" README,
// "Asymmetric Memory Path": weights stay in CPU DRAM and the GPU fetches them
// in-kernel, no staging copy in HBM).  The pointers must be pinned host
// allocations (cudaHostAlloc / cudaHostRegister); a pointer the driver cannot
// map is rejected.
bsf_status resolve_b(int flags, const uint8_t** b, const int32_t** sfb) {
  if (!(flags & BSF_B_HOST_MAPPED)) return BSF_OK;
  void* db = nullptr;
  void* ds = nullptr;
  if (cudaHostGetDevicePointer(&db, const_cast<uint8_t*>(*b), 0) != cudaSuccess ||
      cudaHostGetDevicePointer(&ds, const_cast<int32_t*>(*sfb), 0) != cudaSuccess) {
    cudaGetLastError();   // clear the sticky-free error of the failed query
    return BSF_ERR_INVALID_ARGUMENT;
  }
  *b = static_cast<const uint8_t*>(db);
  *sfb = static_cast<const int32_t*>(ds);
  return BSF_OK;
}

bsf_status check_common(const uint8_t* a, const int32_t* sfa, int64_t sfa_ld, int64_t m_rows, const uint8_t* b,
                        const int32_t* sfb, const void* d, int64_t E, int64_t N, int64_t K, int flags,
                        bool nvfp4 = false) {
  if (E <= 0 || E > kMaxExperts || N <= 0 || K <= 0 || N % 128 || K % 128) return BSF_ERR_INVALID_ARGUMENT;
  if (nvfp4 && K % 256) return BSF_ERR_INVALID_ARGUMENT;
  if (nvfp4 && E > kNvfp4MaxE) return BSF_ERR_UNSUPPORTED;
  if (flags & ~(BSF_B_HOST_MAPPED | BSF_B_TILED | BSF_DEBUG_WITHHOLD_LOADS)) return BSF_ERR_INVALID_ARGUMENT;
  if (!a || !sfa || !b || !sfb || !d) return BSF_ERR_INVALID_ARGUMENT;
  if (sfa_ld < m_rows || sfa_ld % 4) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(a) || !aligned16(b) || !aligned16(d) || !aligned16(sfa) || !aligned16(sfb))
    return BSF_ERR_MISALIGNED;
  if (m_rows > INT32_MAX || E * N > INT32_MAX || K > (1 << 24)) return BSF_ERR_UNSUPPORTED;
  return BSF_OK;
}

}  // namespace
}  // namespace bsf

using namespace bsf;

extern "C" bsf_status bsf_grouped_gemm_contig(const uint8_t* a, const int32_t* sfa, int64_t sfa_ld, int64_t m_cap,
                                              const uint8_t* b, const int32_t* sfb, void* d,
                                              const int32_t* seg_start, const int32_t* counts, int64_t E, int64_t N,
                                              int64_t K, int flags, bsf_stream_t stream) {
  if (m_cap <= 0) return m_cap == 0 ? BSF_OK : BSF_ERR_INVALID_ARGUMENT;
  bsf_status st = check_common(a, sfa, sfa_ld, m_cap, b, sfb, d, E, N, K, flags);
  if (st != BSF_OK) return st;
  if (!seg_start || !counts) return BSF_ERR_INVALID_ARGUMENT;
  if ((st = resolve_b(flags, &b, &sfb)) != BSF_OK) return st;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  GemmArgs args{seg_start, counts, 0, m_cap, sfa, sfa_ld, sfb, static_cast<uint16_t*>(d),
                static_cast<int>(E), static_cast<int>(N), static_cast<int>(K), err,
                flags};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (flags & BSF_B_HOST_MAPPED) {   // one tile per (expert, N-tile) up to 448 rows: weights cross the link once
    const int64_t max_tiles = (m_cap / kHostTok + E) * (N / 128);
    return launch<kHostTok>(args, a, b, max_tiles, s);
  }
  if (N % 256 == 0) {   // 256-row items (two weight tiles), one CTA per SM
    if (E <= 256) {      // 256 x 160 items, four stages
      const int64_t max_items = (m_cap / kWideTok + E) * (N / 256);
      return launch<kWideTok, 1, 256, kFmtFp8, 2>(args, a, b, max_items, s);
    }
    const int64_t max_items = (m_cap / kBigTok + E) * (N / 256);
    return launch<kBigTok, 1, kMaxExperts, kFmtFp8, 2>(args, a, b, max_items, s);
  }
  const int64_t max_tiles = (m_cap / kBigTok + E) * (N / 128);
  return launch<kBigTok, 2>(args, a, b, max_tiles, s);
}

extern "C" bsf_status bsf_grouped_gemm_masked(const uint8_t* a, const int32_t* sfa, int64_t sfa_ld, const uint8_t* b,
                                              const int32_t* sfb, void* d, const int32_t* masked_m, int64_t E,
                                              int64_t max_m, int64_t N, int64_t K, int64_t expected_m, int flags,
                                              bsf_stream_t stream) {
  if (max_m <= 0) return BSF_ERR_INVALID_ARGUMENT;
  const int64_t m_rows = E * max_m;
  bsf_status st = check_common(a, sfa, sfa_ld, m_rows, b, sfb, d, E, N, K, flags);
  if (st != BSF_OK) return st;
  if (!masked_m) return BSF_ERR_INVALID_ARGUMENT;
  if ((st = resolve_b(flags, &b, &sfb)) != BSF_OK) return st;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  GemmArgs args{nullptr, masked_m, max_m, m_rows, sfa, sfa_ld, sfb, static_cast<uint16_t*>(d),
                static_cast<int>(E), static_cast<int>(N), static_cast<int>(K), err,
                flags};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t hint = expected_m > 0 ? expected_m : max_m;
  const bool host = (flags & BSF_B_HOST_MAPPED) != 0;
  // small slots (or, with weights in HBM, small typical counts): the 64-token variant with its deep ring;
  // weights in host memory: the smallest variant that holds a whole slot, so weights cross the link once
  if (max_m <= 64 || (!host && hint <= 32)) {
    const int64_t max_tiles = E * ((max_m + 63) / 64) * (N / 128);
    if (E <= 256) return launch<64, 2, 256>(args, a, b, max_tiles, s);
    return launch<64, 2>(args, a, b, max_tiles, s);
  }
  if (host && max_m > kBigTok) {
    const int64_t max_tiles = E * ((max_m + kHostTok - 1) / kHostTok) * (N / 128);
    return launch<kHostTok>(args, a, b, max_tiles, s);
  }
  if (N % 256 == 0) {
    if (E <= 256) {
      const int64_t max_items = E * ((max_m + kWideTok - 1) / kWideTok) * (N / 256);
      return launch<kWideTok, 1, 256, kFmtFp8, 2>(args, a, b, max_items, s);
    }
    const int64_t max_items = E * ((max_m + kBigTok - 1) / kBigTok) * (N / 256);
    return launch<kBigTok, 1, kMaxExperts, kFmtFp8, 2>(args, a, b, max_items, s);
  }
  const int64_t max_tiles = E * ((max_m + kBigTok - 1) / kBigTok) * (N / 128);
  return launch<kBigTok, 2>(args, a, b, max_tiles, s);
}

// ---------------------------------------------------------------- NVFP4
// Same kernel with E2M1 operands and UE4M3 scales per 16 K ("AsymGEMM"
// README, "FP4 Asymmetric GEMM"; block-scaled MMA kind::mxf4nvf4).

extern "C" bsf_status bsf_grouped_gemm_nvfp4_contig(const uint8_t* a, const int32_t* sfa, int64_t sfa_ld,
                                                    int64_t m_cap, int a_exp, const uint8_t* b, const int32_t* sfb,
                                                    const int32_t* b_exp, void* d, const int32_t* seg_start,
                                                    const int32_t* counts, int64_t E, int64_t N, int64_t K,
                                                    int flags, bsf_stream_t stream) {
  if (m_cap <= 0) return m_cap == 0 ? BSF_OK : BSF_ERR_INVALID_ARGUMENT;
  if (a_exp < -100 || a_exp > 100) return BSF_ERR_INVALID_ARGUMENT;
  bsf_status st = check_common(a, sfa, sfa_ld, m_cap, b, sfb, d, E, N, K, flags, true);
  if (st != BSF_OK) return st;
  if (!seg_start || !counts) return BSF_ERR_INVALID_ARGUMENT;
  if ((st = resolve_b(flags, &b, &sfb)) != BSF_OK) return st;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  GemmArgs args{seg_start, counts, 0, m_cap, sfa, sfa_ld, sfb, static_cast<uint16_t*>(d),
                static_cast<int>(E), static_cast<int>(N), static_cast<int>(K), err,
                flags, a_exp, b_exp};
  if (N % 256 == 0) {   // 256 x 192 items (two weight tiles), one CTA per SM
    const int64_t max_items = (m_cap / 192 + E) * (N / 256);
    return launch<192, 1, kNvfp4MaxE, kFmtNvfp4, 2>(args, a, b, max_items, reinterpret_cast<cudaStream_t>(stream));
  }
  const int64_t max_tiles = (m_cap / 128 + E) * (N / 128);
  return launch<128, 2, kNvfp4MaxE, kFmtNvfp4>(args, a, b, max_tiles, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" bsf_status bsf_grouped_gemm_nvfp4_masked(const uint8_t* a, const int32_t* sfa, int64_t sfa_ld, int a_exp,
                                                    const uint8_t* b, const int32_t* sfb, const int32_t* b_exp,
                                                    void* d, const int32_t* masked_m, int64_t E, int64_t max_m,
                                                    int64_t N, int64_t K, int64_t expected_m, int flags,
                                                    bsf_stream_t stream) {
  if (max_m <= 0) return BSF_ERR_INVALID_ARGUMENT;
  if (a_exp < -100 || a_exp > 100) return BSF_ERR_INVALID_ARGUMENT;
  const int64_t m_rows = E * max_m;
  bsf_status st = check_common(a, sfa, sfa_ld, m_rows, b, sfb, d, E, N, K, flags, true);
  if (st != BSF_OK) return st;
  if (!masked_m) return BSF_ERR_INVALID_ARGUMENT;
  if ((st = resolve_b(flags, &b, &sfb)) != BSF_OK) return st;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  GemmArgs args{nullptr, masked_m, max_m, m_rows, sfa, sfa_ld, sfb, static_cast<uint16_t*>(d),
                static_cast<int>(E), static_cast<int>(N), static_cast<int>(K), err,
                flags, a_exp, b_exp};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t hint = expected_m > 0 ? expected_m : max_m;
  if (max_m <= 64 || ((flags & BSF_B_HOST_MAPPED) == 0 && hint <= 32)) {
    const int64_t max_tiles = E * ((max_m + 63) / 64) * (N / 128);
    return launch<64, 2, kNvfp4MaxE, kFmtNvfp4>(args, a, b, max_tiles, s);
  }
  if (N % 256 == 0) {
    const int64_t max_items = E * ((max_m + 191) / 192) * (N / 256);
    return launch<192, 1, kNvfp4MaxE, kFmtNvfp4, 2>(args, a, b, max_items, s);
  }
  const int64_t max_tiles = E * ((max_m + 127) / 128) * (N / 128);
  return launch<128, 2, kNvfp4MaxE, kFmtNvfp4>(args, a, b, max_tiles, s);
}

// ---------------------------------------------------------------- BF16
// Same kernel on unquantised bf16 operands ("AsymGEMM" README, "BF16 Asymmetric
// GEMM"): kind::f16 MMA with both operands BF16, FP32 accumulation, no scales.

namespace bsf {
namespace {

bsf_status check_bf16(const void* a, int64_t m_rows, const void* b, const void* d, int64_t E, int64_t N, int64_t K,
                      int flags, const uint8_t** b_dev) {
  if (E <= 0 || E > kMaxExperts || N <= 0 || K <= 0 || N % 128 || K % 64) return BSF_ERR_INVALID_ARGUMENT;
  if (flags & ~(BSF_B_HOST_MAPPED | BSF_B_TILED | BSF_DEBUG_WITHHOLD_LOADS)) return BSF_ERR_INVALID_ARGUMENT;
  if (!a || !b || !d) return BSF_ERR_INVALID_ARGUMENT;
  if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return BSF_ERR_MISALIGNED;
  if (m_rows > INT32_MAX || E * N > INT32_MAX || K > (1 << 23)) return BSF_ERR_UNSUPPORTED;
  *b_dev = static_cast<const uint8_t*>(b);
  if (flags & BSF_B_HOST_MAPPED) {
    void* db = nullptr;
    if (cudaHostGetDevicePointer(&db, const_cast<void*>(b), 0) != cudaSuccess) {
      cudaGetLastError();
      return BSF_ERR_INVALID_ARGUMENT;
    }
    *b_dev = static_cast<const uint8_t*>(db);
  }
  return BSF_OK;
}

}  // namespace
}  // namespace bsf

extern "C" bsf_status bsf_grouped_gemm_bf16_contig(const void* a, int64_t m_cap, const void* b, void* d,
                                                   const int32_t* seg_start, const int32_t* counts, int64_t E,
                                                   int64_t N, int64_t K, int flags, bsf_stream_t stream) {
  if (m_cap <= 0) return m_cap == 0 ? BSF_OK : BSF_ERR_INVALID_ARGUMENT;
  const uint8_t* bd = nullptr;
  bsf_status st = check_bf16(a, m_cap, b, d, E, N, K, flags, &bd);
  if (st != BSF_OK) return st;
  if (!seg_start || !counts) return BSF_ERR_INVALID_ARGUMENT;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  GemmArgs args{seg_start, counts, 0, m_cap, nullptr, 0, nullptr, static_cast<uint16_t*>(d),
                static_cast<int>(E), static_cast<int>(N), static_cast<int>(K), err,
                flags};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* ad = static_cast<const uint8_t*>(a);
  if (flags & BSF_B_HOST_MAPPED) {
    const int64_t max_tiles = (m_cap / kHostTok + E) * (N / 128);
    return launch<kHostTok, 1, kMaxExperts, kFmtBf16>(args, ad, bd, max_tiles, s);
  }
  if (N % 256 == 0) {   // 256-row items (two weight tiles), one CTA per SM
    if (E <= 256) {      // 256 x 160 items, four stages
      const int64_t max_items = (m_cap / kWideTok + E) * (N / 256);
      return launch<kWideTok, 1, 256, kFmtBf16, 2>(args, ad, bd, max_items, s);
    }
    const int64_t max_items = (m_cap / kBigTok + E) * (N / 256);
    return launch<kBigTok, 1, kMaxExperts, kFmtBf16, 2>(args, ad, bd, max_items, s);
  }
  const int64_t max_tiles = (m_cap / kBigTok + E) * (N / 128);
  return launch<kBigTok, 2, kMaxExperts, kFmtBf16>(args, ad, bd, max_tiles, s);
}

extern "C" bsf_status bsf_grouped_gemm_bf16_masked(const void* a, const void* b, void* d, const int32_t* masked_m,
                                                   int64_t E, int64_t max_m, int64_t N, int64_t K,
                                                   int64_t expected_m, int flags, bsf_stream_t stream) {
  if (max_m <= 0) return BSF_ERR_INVALID_ARGUMENT;
  const int64_t m_rows = E * max_m;
  const uint8_t* bd = nullptr;
  bsf_status st = check_bf16(a, m_rows, b, d, E, N, K, flags, &bd);
  if (st != BSF_OK) return st;
  if (!masked_m) return BSF_ERR_INVALID_ARGUMENT;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  GemmArgs args{nullptr, masked_m, max_m, m_rows, nullptr, 0, nullptr, static_cast<uint16_t*>(d),
                static_cast<int>(E), static_cast<int>(N), static_cast<int>(K), err,
                flags};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* ad = static_cast<const uint8_t*>(a);
  const int64_t hint = expected_m > 0 ? expected_m : max_m;
  const bool host = (flags & BSF_B_HOST_MAPPED) != 0;
  if (max_m <= 64 || (!host && hint <= 32)) {
    const int64_t max_tiles = E * ((max_m + 63) / 64) * (N / 128);
    if (E <= 256) return launch<64, 2, 256, kFmtBf16>(args, ad, bd, max_tiles, s);
    return launch<64, 2, kMaxExperts, kFmtBf16>(args, ad, bd, max_tiles, s);
  }
  if (host && max_m > kBigTok) {
    const int64_t max_tiles = E * ((max_m + kHostTok - 1) / kHostTok) * (N / 128);
    return launch<kHostTok, 1, kMaxExperts, kFmtBf16>(args, ad, bd, max_tiles, s);
  }
  if (N % 256 == 0) {
    if (E <= 256) {
      const int64_t max_items = E * ((max_m + kWideTok - 1) / kWideTok) * (N / 256);
      return launch<kWideTok, 1, 256, kFmtBf16, 2>(args, ad, bd, max_items, s);
    }
    const int64_t max_items = E * ((max_m + kBigTok - 1) / kBigTok) * (N / 256);
    return launch<kBigTok, 1, kMaxExperts, kFmtBf16, 2>(args, ad, bd, max_items, s);
  }
  const int64_t max_tiles = E * ((max_m + kBigTok - 1) / kBigTok) * (N / 128);
  return launch<kBigTok, 2, kMaxExperts, kFmtBf16>(args, ad, bd, max_tiles, s);
}

// ---------------------------------------------------------------- FP8 with float32 scales
// "AsymGEMM" README, disable_ue8m0_cast: the scales stay float32.  They cannot
// feed the block-scaled MMA (UE8M0 / UE4M3 only), so each 128-K stage is a
// separate unscaled MMA (kind::f8f6f4) into a TMEM partial, and the epilogue
// warps add sA * sB * partial in FP32 (the DeepGEMM article's software path of
// "补偿机制二").

extern "C" bsf_status bsf_grouped_gemm_f32sf_contig(const uint8_t* a, const float* sfa, int64_t sfa_ld, int64_t m_cap,
                                                    const uint8_t* b, const float* sfb, void* d,
                                                    const int32_t* seg_start, const int32_t* counts, int64_t E,
                                                    int64_t N, int64_t K, int flags, bsf_stream_t stream) {
  if (m_cap <= 0) return m_cap == 0 ? BSF_OK : BSF_ERR_INVALID_ARGUMENT;
  const int32_t* sfa_i = reinterpret_cast<const int32_t*>(sfa);
  const int32_t* sfb_i = reinterpret_cast<const int32_t*>(sfb);
  bsf_status st = check_common(a, sfa_i, sfa_ld, m_cap, b, sfb_i, d, E, N, K, flags);
  if (st != BSF_OK) return st;
  if (!seg_start || !counts) return BSF_ERR_INVALID_ARGUMENT;
  if ((st = resolve_b(flags, &b, &sfb_i)) != BSF_OK) return st;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  GemmArgs args{seg_start, counts, 0, m_cap, nullptr, sfa_ld, nullptr, static_cast<uint16_t*>(d),
                static_cast<int>(E), static_cast<int>(N), static_cast<int>(K), err,
                flags, 0, nullptr, sfa, reinterpret_cast<const float*>(sfb_i)};
  // 128-token tiles: each weight tile is streamed once per 128 rows of an expert
  const int64_t max_tiles = (m_cap / 128 + E) * (N / 128);
  return launch<128, 1, kMaxExperts, kFmtFp8F32>(args, a, b, max_tiles, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" bsf_status bsf_grouped_gemm_f32sf_masked(const uint8_t* a, const float* sfa, int64_t sfa_ld,
                                                    const uint8_t* b, const float* sfb, void* d,
                                                    const int32_t* masked_m, int64_t E, int64_t max_m, int64_t N,
                                                    int64_t K, int64_t expected_m, int flags, bsf_stream_t stream) {
  if (max_m <= 0) return BSF_ERR_INVALID_ARGUMENT;
  const int64_t m_rows = E * max_m;
  const int32_t* sfa_i = reinterpret_cast<const int32_t*>(sfa);
  const int32_t* sfb_i = reinterpret_cast<const int32_t*>(sfb);
  bsf_status st = check_common(a, sfa_i, sfa_ld, m_rows, b, sfb_i, d, E, N, K, flags);
  if (st != BSF_OK) return st;
  if (!masked_m) return BSF_ERR_INVALID_ARGUMENT;
  if ((st = resolve_b(flags, &b, &sfb_i)) != BSF_OK) return st;
  int* err = device_error_ptr();
  if (!err) return BSF_ERR_CUDA;
  GemmArgs args{nullptr, masked_m, max_m, m_rows, nullptr, sfa_ld, nullptr, static_cast<uint16_t*>(d),
                static_cast<int>(E), static_cast<int>(N), static_cast<int>(K), err,
                flags, 0, nullptr, sfa, reinterpret_cast<const float*>(sfb_i)};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // small slots or small typical counts: 32-token tiles, two CTAs per SM (32 accumulators per thread);
  // same-box A/B at decode: 258 us against 329 us for the 64-token tile with one CTA per SM
  const int64_t hint = expected_m > 0 ? expected_m : max_m;
  if (max_m <= 32 || hint <= 16) {
    const int64_t max_tiles = E * ((max_m + 31) / 32) * (N / 128);
    if (E <= 256) return launch<32, 2, 256, kFmtFp8F32>(args, a, b, max_tiles, s);
    return launch<32, 2, kMaxExperts, kFmtFp8F32>(args, a, b, max_tiles, s);
  }
  if (max_m <= 64 || hint <= 64) {
    const int64_t max_tiles = E * ((max_m + 63) / 64) * (N / 128);
    return launch<64, 1, kMaxExperts, kFmtFp8F32>(args, a, b, max_tiles, s);
  }
  const int64_t max_tiles = E * ((max_m + 127) / 128) * (N / 128);
  return launch<128, 1, kMaxExperts, kFmtFp8F32>(args, a, b, max_tiles, s);
}
