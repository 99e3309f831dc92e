/*
 * bsfroute — FP8 block-scaled MoE routing + grouped GEMM for GB300 (sm_103a).
 *
 * C ABI of the hot path:
 *   quantise_act  -> route (+ scatter) -> grouped_gemm_{contig,masked} -> combine
 * plus the once-per-weight-load steps quantise_weight and prepare_weight_sf,
 * and for small batches dispatch (quantise + route + scatter in one launch).
 * The same path on the pages' other operand formats, declared further down:
 *   NVFP4  (E2M1 + one UE4M3 scale per 16 values, *_nvfp4),
 *   BF16   (unquantised, *_bf16),
 *   FP8 with float32 scale factors (*_f32sf).
 *
 * Conventions of every entry point
 *   - Pointers are DEVICE pointers (CUDA global memory) unless a parameter says
 *     otherwise.  The caller allocates and owns every buffer; no entry point
 *     allocates memory.
 *   - `stream` is a cudaStream_t (0 = legacy default stream).  All work is
 *     enqueued on it; calls never synchronise the device.
 *   - Arguments are validated on the host before anything is enqueued; a bad
 *     argument returns a non-zero bsf_status and enqueues nothing.  Sizes
 *     beyond any real problem (more than 2^31 - 1 rows, tokens or experts x
 *     weight rows, or rows wider than 2^24 elements or bytes) return
 *     BSF_ERR_UNSUPPORTED before any product of them is formed.
 *   - Problems found while the kernels run (an expert id >= E, a masked slot
 *     overflow, a weight scale that is not a power of two, a wait that ran
 *     out) set bits of a sticky device error word; read it with
 *     bsf_get_device_error.
 *   - bf16 is IEEE bfloat16 stored as uint16; e4m3 is FP8 E4M3 ("e4m3fn":
 *     bias 7, max 448, no infinities) stored as uint8.
 *
 * Scale-factor (SF) format (DeepGEMM FP8 article, nxmr.cn, sections
 * "补偿机制一" and "补偿机制三"): every scale is an exact power of two 2**e,
 * stored as a UE8M0 byte e + 127; four bytes are packed per int32, byte j
 * (bits 8j..8j+7) holding K-block 4i + j of word i (K-blocks of 128).  Packed
 * SF tensors are MN-major: element [i][row] at offset i * ld + row, with ld
 * (in int32 words) a multiple of 4 (16 bytes, the TMA-aligned stride).
 */
#ifndef BSFROUTE_H
#define BSFROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bsf_stream_t; /* same type as cudaStream_t */

typedef enum bsf_status {
  BSF_OK = 0,
  BSF_ERR_INVALID_ARGUMENT = 1, /* a size, layout or pointer is not acceptable */
  BSF_ERR_MISALIGNED = 2,       /* a pointer or stride breaks the 16-byte TMA alignment */
  BSF_ERR_UNSUPPORTED = 3,      /* the shape is valid but not supported by this build */
  BSF_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed */
  BSF_ERR_DEVICE = 5            /* the current device is not an sm_100-class GPU */
} bsf_status;

/* Device error word bits (sticky until cleared). */
#define BSF_DEVERR_EXPERT_ID 0x1       /* a topk id >= E was seen (route skips it) */
#define BSF_DEVERR_MASKED_OVERFLOW 0x2 /* masked layout: assignments past max_m were dropped */
#define BSF_DEVERR_TIMEOUT 0x4         /* a bounded wait ran out; the kernel returned early */
#define BSF_DEVERR_BAD_SCALE 0x8       /* a weight scale is not a positive power of two */
#define BSF_DEVERR_SEGMENT 0x10        /* a segment does not fit the A buffer; it was skipped */

/* Layouts of the packed token operand ("AsymGEMM" README, "Token Layout Protocols"). */
#define BSF_LAYOUT_CONTIGUOUS 0
#define BSF_LAYOUT_MASKED 1

/* GEMM flags. */
#define BSF_B_HOST_MAPPED 0x1 /* b / sfb are host pointers to pinned, mapped host memory */
/* b holds the weights in the tiled layout written by bsf_tile_weights (any
 * operand format; scale factors are unchanged).  Every 128-row x 128-byte
 * block the kernel loads is then one contiguous 16 KB run of memory instead
 * of 128 strided 128-byte pieces: fewer DRAM pages per load, measured 4%
 * faster on the weight-streaming decode GEMM.  Combines with
 * BSF_B_HOST_MAPPED. */
#define BSF_B_TILED 0x2
/* Fault injection for tests of the failure path: the kernel's load producer
 * withholds every load, so each consumer's bounded wait runs out; the kernel
 * sets BSF_DEVERR_TIMEOUT, releases its tensor memory and returns without
 * writing d.  No GPU fault or hang is involved. */
#define BSF_DEBUG_WITHHOLD_LOADS 0x100

const char* bsf_status_string(bsf_status status);
int bsf_version(void);

/* Reads the device error word into *code (host pointer) after synchronising
 * `stream`; clears it when `clear` is non-zero. */
bsf_status bsf_get_device_error(int32_t* code, int clear, bsf_stream_t stream);

/*
 * bsf_quantise_act — activations to FP8 with 1 x 128 power-of-two scales.
 * DeepGEMM article "补偿机制一" (power-of-two SF, UE8M0) and "FP8 的精度陷阱"
 * (E4M3); recipe (gran_m, gran_k) = (1, 128).
 *   x     bf16  [T, K] row-major.
 *   q     e4m3  [T, K] row-major (output).
 *   sf    int32 [ceil(K/512)][sf_ld] packed MN-major (output); rows >= T are
 *         not written.  sf_ld >= T, multiple of 4.
 * For each row t and K-block b: amax = max |x|; e = least integer with
 * amax <= 448 * 2**e (0 for an all-zero block), clamped to [-126, 127];
 * q = E4M3_RNE_satfinite(x * 2**-e); SF byte e + 127.
 * Needs K % 128 == 0, T >= 0.  T == 0 is a no-op.
 */
bsf_status bsf_quantise_act(const void* x, int64_t T, int64_t K, uint8_t* q, int32_t* sf, int64_t sf_ld,
                            bsf_stream_t stream);

/*
 * bsf_quantise_act_rows — bsf_quantise_act on the routed rows of a packed
 * operand only (e.g. the input of a second grouped GEMM that shares the
 * routing): row t is quantised iff t < *rows_used and token_of_row[t] >= 0,
 * with token_of_row and rows_used = seg_start + E from bsf_route.  The other
 * rows (segment padding, rows past the last segment) of q and sf are not
 * written: no stored GEMM output depends on them ("GEMM 执行方式" §4.6 leaves
 * padding rows uninitialised).  Same arithmetic, layout and checks as
 * bsf_quantise_act; token_of_row int32 [T] and rows_used int32 [1] are device
 * pointers.
 */
bsf_status bsf_quantise_act_rows(const void* x, int64_t T, int64_t K, const int32_t* token_of_row,
                                 const int32_t* rows_used, uint8_t* q, int32_t* sf, int64_t sf_ld,
                                 bsf_stream_t stream);

/*
 * bsf_quantise_weight — expert weights to FP8 with 128 x 128 power-of-two scales
 * (same rule as bsf_quantise_act over 128 x 128 blocks; recipe gran_n = 128).
 *   w      bf16  [E, N, K] row-major.
 *   q      e4m3  [E, N, K] (output).
 *   sf128  fp32  [E, N/128, K/128] (output), every entry 2**e.
 * Needs N % 128 == 0, K % 128 == 0.
 */
bsf_status bsf_quantise_weight(const void* w, int64_t E, int64_t N, int64_t K, uint8_t* q, float* sf128,
                               bsf_stream_t stream);

/*
 * bsf_prepare_weight_sf — once per weight load: fp32 128 x 128 scales to the
 * per-row packed UE8M0 layout the GEMM reads (DeepGEMM article "补偿机制三":
 * weight SFs are transformed once and reused).
 *   sf128  fp32  [E, N/128, K/128], each a positive power of two.
 *   sfb    int32 [E][ceil(K/512)][N] (output): word [e][i][n] packs the bytes
 *          of K-blocks 4i..4i+3 of row block n / 128; bytes past K/128 are 127.
 * A scale that is not a power of two sets BSF_DEVERR_BAD_SCALE (its byte is
 * written as 127).
 */
bsf_status bsf_prepare_weight_sf(const float* sf128, int64_t E, int64_t N, int64_t K, int32_t* sfb,
                                 bsf_stream_t stream);

/*
 * bsf_route — top-k routing, segment offsets, inverse index, and (optionally)
 * the scatter of quantised rows into the packed operand.
 * "GEMM 执行方式" (rainlin-net) §4.2 (topk tensors, R = T k_r = sum M_e),
 * §4.3 (packed layout, m_indices, output_index), §4.6 (A-aligned segments,
 * ep_scatter); "CuTeDSL bei Perplexity", MoE dispatch (count per expert,
 * unique index per token, copy into optionally padded buffers).
 *   topk_ids      int32 [T, kr]; ids < 0 are dropped routes; ids >= E set
 *                 BSF_DEVERR_EXPERT_ID and are dropped.
 *   layout        BSF_LAYOUT_CONTIGUOUS: segment e spans
 *                 [seg_start[e], seg_start[e+1]), length ceil(M_e/align)*align;
 *                 BSF_LAYOUT_MASKED: segment e spans [e*max_m, (e+1)*max_m),
 *                 at most max_m rows, further assignments dropped
 *                 (BSF_DEVERR_MASKED_OVERFLOW).
 *   align_or_max_m  align (>= 1) for CONTIGUOUS, max_m (>= 1) for MASKED.
 *   counts        int32 [E] (output): rows placed per expert (M_e, or
 *                 min(M_e, max_m) for MASKED) — the GEMM's counts / masked_m.
 *   seg_start     int32 [E+1] (output).
 *   output_index  int32 [T, kr] (output): packed row of each assignment, -1 if dropped.
 *   token_of_row  int32 [m_cap] (output): token of each packed row, -1 for
 *                 padding rows; rows >= seg_start[E] are not written.
 *   m_indices     int32 [m_cap] (output, may be NULL): expert owning each
 *                 packed row < seg_start[E] (padding rows included).
 *   m_cap         rows of the packed buffers: at least T*kr + E*(align-1)
 *                 (CONTIGUOUS) or E*max_m (MASKED) — no device-to-host sync
 *                 is needed to size them.
 *   q, sf, sf_ld  optional scatter source (NULL: indices only): e4m3 [T, K]
 *                 and packed SF [ceil(K/512)][sf_ld] from bsf_quantise_act.
 *   a_packed      e4m3 [m_cap, K] (output): row r = q[token_of_row[r]];
 *                 padding rows are not written (uninitialised, as in §4.6;
 *                 no GEMM output row that is stored depends on them).
 *   sfa_packed    int32 [ceil(K/512)][sfa_ld] (output), sfa_ld >= m_cap,
 *                 multiple of 4; padding rows are not written.
 *   workspace     device scratch of bsf_route_workspace_bytes(T, kr, E) bytes
 *                 (that function returns 0 for sizes bsf_route rejects:
 *                 T < 0, kr <= 0, E <= 0, or T * kr above INT32_MAX).
 * Order inside an expert: ascending flat index t*kr + r (stable; the order of
 * the worked example in §4.3 / §4.6).  Deterministic.
 */
size_t bsf_route_workspace_bytes(int64_t T, int64_t kr, int64_t E);
bsf_status bsf_route(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout, int64_t align_or_max_m,
                     int32_t* counts, int32_t* seg_start, int32_t* output_index, int32_t* token_of_row,
                     int32_t* m_indices, int64_t m_cap, const uint8_t* q, const int32_t* sf, int64_t sf_ld,
                     int64_t K, uint8_t* a_packed, int32_t* sfa_packed, int64_t sfa_ld, void* workspace,
                     size_t workspace_bytes, bsf_stream_t stream);

/*
 * bsf_route_quantise — bsf_quantise_act + bsf_route with the scatter, fused
 * for batches of any size: route (as bsf_route), then one warp per (token,
 * 512-wide K group) reads the token's bf16 row segment ONCE, quantises it
 * (the same arithmetic and bytes as bsf_quantise_act) and writes the codes
 * and the scale word to each of the token's k_r packed rows.  The token-major
 * q / sf copies are neither written nor re-read.
 * "GEMM 执行方式" §4.2-§4.6 (routing, packed layout, ep_scatter);
 * "CuTeDSL bei Perplexity", MoE dispatch (quantise and copy in one pass);
 * DeepGEMM article "补偿机制一" (1 x 128 UE8M0 block scales).
 *   x             bf16 [T, K], K % 128 == 0 (device, caller-owned, read only).
 *   a_packed      e4m3 [m_cap, K], sfa_packed int32 [ceil(K/512)][sfa_ld],
 *                 sfa_ld >= m_cap and a multiple of 4 (outputs): routed rows
 *                 written, padding rows left as they were.
 *   kr <= 32 (else BSF_ERR_UNSUPPORTED).  x, a_packed and sfa_packed must be
 *   16-byte aligned (BSF_ERR_MISALIGNED).
 *   Every other argument, output, device error bit and host-side check as in
 *   bsf_route; every output is bit-identical to bsf_quantise_act followed by
 *   bsf_route with the scatter.  Nothing is allocated; asynchronous on stream.
 */
bsf_status bsf_route_quantise(const void* x, int64_t T, int64_t K, const int32_t* topk_ids, int64_t kr, int64_t E,
                              int layout, int64_t align_or_max_m, int32_t* counts, int32_t* seg_start,
                              int32_t* output_index, int32_t* token_of_row, int32_t* m_indices, int64_t m_cap,
                              uint8_t* a_packed, int32_t* sfa_packed, int64_t sfa_ld, void* workspace,
                              size_t workspace_bytes, bsf_stream_t stream);

/*
 * bsf_route_no_alloc — bsf_route without a caller-provided workspace.
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot call cudaMalloc where they route: serving runtimes that reserve
 * all device memory at start-up and hand the library only its inputs and
 * outputs (cudaMalloc would fail or fragment their pool, and it synchronises
 * the device, stalling every other stream), plug-ins whose host framework owns
 * the allocator and forbids direct device allocation, and code running inside
 * an allocator callback or memory-pressure handler, where allocating again
 * could re-enter the allocator.
 * Same arguments, outputs and errors as bsf_route minus workspace /
 * workspace_bytes (T * kr above INT32_MAX is BSF_ERR_UNSUPPORTED).  The scratch is a file-scope device array of
 * BSF_ROUTE_STATIC_SCRATCH_BYTES bytes (256 KiB) that every GPU which loads
 * the library holds until the process exits; a problem whose
 * bsf_route_workspace_bytes(T, kr, E) exceeds it is rejected with
 * BSF_ERR_UNSUPPORTED before anything is enqueued.  The first call on a
 * device resolves the array's device address (cudaGetSymbolAddress, with that
 * device current), so make that first call before any stream capture.
 * Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 * All calls on a device share that device's one array, so calls that
 * overlap on the GPU (for instance on two streams of the same device) race
 * with each other: order them on one stream.  The array keeps the last call's
 * contents; every word a call reads is first written by that same call.
 */
#define BSF_ROUTE_STATIC_SCRATCH_BYTES (256 * 1024)
bsf_status bsf_route_no_alloc(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout,
                              int64_t align_or_max_m, int32_t* counts, int32_t* seg_start, int32_t* output_index,
                              int32_t* token_of_row, int32_t* m_indices, int64_t m_cap, const uint8_t* q,
                              const int32_t* sf, int64_t sf_ld, int64_t K, uint8_t* a_packed, int32_t* sfa_packed,
                              int64_t sfa_ld, bsf_stream_t stream);

/*
 * bsf_dispatch — quantise + route + scatter in ONE launch, for small batches
 * (decode): T*kr <= BSF_DISPATCH_MAX_ASSIGNMENTS and E <=
 * BSF_DISPATCH_MAX_EXPERTS, else BSF_ERR_UNSUPPORTED (use bsf_quantise_act +
 * bsf_route).
 * "CuTeDSL bei Perplexity", MoE dispatch (decode: one block holds all the
 * routing information; routing and copies in one launch).  Every CTA routes
 * the whole batch in shared memory, then quantises its share of the routed
 * rows straight from x into their packed rows, so no grid-wide barrier is
 * needed.  Outputs are bit-identical to bsf_quantise_act followed by
 * bsf_route with the scatter (same arguments and layouts as those two; the
 * token-major q / sf copies are not produced).
 *   x             bf16 [T, K], K % 128 == 0 (device, caller-owned, read only).
 *   a_packed      e4m3 [m_cap, K]; sfa_packed int32 [ceil(K/512)][sfa_ld]
 *                 (device, caller-owned): routed rows written, padding rows
 *                 left as they were.
 *   other arguments, the device error bits (EXPERT_ID, MASKED_OVERFLOW,
 *   SEGMENT) and the host-side checks are as in bsf_route; x, a_packed and
 *   sfa_packed must be 16-byte aligned (BSF_ERR_MISALIGNED).  Nothing is
 *   allocated; the call is asynchronous on `stream`.
 */
#define BSF_DISPATCH_MAX_ASSIGNMENTS 16384
#define BSF_DISPATCH_MAX_EXPERTS 256
bsf_status bsf_dispatch(const void* x, int64_t T, int64_t K, const int32_t* topk_ids, int64_t kr, int64_t E,
                        int layout, int64_t align_or_max_m, int32_t* counts, int32_t* seg_start,
                        int32_t* output_index, int32_t* token_of_row, int32_t* m_indices, int64_t m_cap,
                        uint8_t* a_packed, int32_t* sfa_packed, int64_t sfa_ld, bsf_stream_t stream);

/*
 * Launch order: every call is stream-ordered.  The small-batch tile
 * (bsf_grouped_gemm_masked with max_m <= 64, or with expected_m <= 32 and
 * device-resident weights) is launched as a programmatic dependent
 * of the preceding kernel on the stream: its CTAs may be scheduled while that
 * kernel drains, and they touch no global memory until it has completed.
 *
 * Tensor memory: every GEMM CTA allocates its tensor-memory columns on entry
 * (tcgen05.alloc), which waits, with no time limit, until an SM has that many
 * columns free.  GEMMs enqueued on two streams of one device can share an SM;
 * a CTA of the second then waits until a CTA of the first exits.  Both finish
 * (every other wait in the kernels is bounded), but they serialise on the SM.
 *
 * bsf_grouped_gemm_contig — D[r, :] = BF16( dequant(A[r, :]) . dequant(B_e)^T )
 * for every expert e and every row r in [seg_start[e], seg_start[e] + counts[e]).
 * "GEMM 执行方式" §4.1 (P independent problems), §4.4 (Y_e = X_e W_e^T);
 * "AsymGEMM" README API reference (m_grouped_fp8_asym_gemm_nt_contiguous:
 * (data, scale) pairs, NT, bf16 output); DeepGEMM article "补偿机制二"
 * (block-scaled MMA consumes the UE8M0 scales).
 *   a        e4m3  [m_cap, K]; sfa int32 [ceil(K/512)][sfa_ld] (1 x 128 SFs).
 *   b        e4m3  [E, N, K]; sfb int32 [E][ceil(K/512)][N] from bsf_prepare_weight_sf.
 *   d        bf16  [m_cap, N] (output); only the rows above are written.
 *   seg_start, counts  int32 [E+1], [E] (device), e.g. from bsf_route.
 * FP32 accumulation on the tensor cores, round-to-nearest-even to bf16.
 * Needs N % 128 == 0, K % 128 == 0, 16-byte aligned a, b, d.
 * flags: BSF_B_HOST_MAPPED — b and sfb live in pinned host memory mapped
 * into the device address space (the "AsymGEMM" asymmetric memory path);
 * the kernel reads them directly, nothing is staged in HBM.  BSF_B_TILED —
 * b is in the layout of bsf_tile_weights (all GEMM entry points accept it).
 */
bsf_status bsf_grouped_gemm_contig(const uint8_t* a, const int32_t* sfa, int64_t sfa_ld, int64_t m_cap,
                                   const uint8_t* b, const int32_t* sfb, void* d, const int32_t* seg_start,
                                   const int32_t* counts, int64_t E, int64_t N, int64_t K, int flags,
                                   bsf_stream_t stream);

/*
 * bsf_grouped_gemm_masked — the same contraction on the masked layout
 * ("AsymGEMM" README, "Token Layout Protocols": expert g at rows g*max_m,
 * masked_m[g] valid rows, 0 = inactive; m_grouped_fp8_asym_gemm_nt_masked).
 *   a    e4m3 [E, max_m, K]; sfa int32 [ceil(K/512)][sfa_ld], sfa_ld >= E*max_m.
 *   d    bf16 [E, max_m, N] (output); rows >= masked_m[g] are not written.
 *   masked_m int32 [E] (device), each <= max_m.
 *   expected_m  hint of the typical masked_m (0: unknown); picks the token tile.
 */
bsf_status bsf_grouped_gemm_masked(const uint8_t* a, const int32_t* sfa, int64_t sfa_ld, const uint8_t* b,
                                   const int32_t* sfb, void* d, const int32_t* masked_m, int64_t E, int64_t max_m,
                                   int64_t N, int64_t K, int64_t expected_m, int flags, bsf_stream_t stream);

/*
 * bsf_tile_weights — rewrites expert weights from row-major [E, N, row_bytes]
 * into the layout BSF_B_TILED names: [E][N/128][row_bytes/128][128][128],
 * i.e. out[((e * N/128 + n / 128) * (row_bytes/128) + c / 128) * 16384
 *          + (n % 128) * 128 + c % 128] = b[(e * N + n) * row_bytes + c]
 * for row n and byte c of expert e.  A byte permutation, the same for every
 * operand format: row_bytes = K (FP8), K / 2 (NVFP4), 2 K (BF16).
 *   b, out  device memory, E * N * row_bytes bytes each, 16-byte aligned,
 *           distinct (tile in HBM, then copy to pinned host memory for
 *           BSF_B_HOST_MAPPED).
 * Needs N % 128 == 0, row_bytes % 128 == 0, E * N * row_bytes / 128 < 2**31.
 * Asynchronous on `stream`; the caller owns both buffers.
 */
bsf_status bsf_tile_weights(const uint8_t* b, int64_t E, int64_t N, int64_t row_bytes, uint8_t* out,
                            bsf_stream_t stream);

/*
 * bsf_combine — weighted un-permute: z[t, :] = BF16( sum_r p[t, r] * y[output_index[t, r], :] )
 * "GEMM 执行方式" §4.4 / §4.6 (ep_gather); "CuTeDSL bei Perplexity" (combine
 * accumulates in registers using the dispatch offsets).
 *   y             bf16  [y_rows, N] expert outputs (the GEMM's d).
 *   output_index  int32 [T, kr] from bsf_route; -1 entries are skipped.
 *   topk_weights  fp32  [T, kr].
 *   z             bf16  [T, N] (output).
 * FP32 accumulation in r order, round-to-nearest-even to bf16.  Needs N % 8 == 0.
 */
bsf_status bsf_combine(const void* y, int64_t y_rows, const int32_t* output_index, const float* topk_weights,
                       int64_t T, int64_t kr, int64_t N, void* z, bsf_stream_t stream);

/*
 * bsf_checksum_u64 — streaming read of `bytes` (multiple of 16) at `p`: *out
 * (device pointer) = XOR of all 64-bit words.  With BSF_B_HOST_MAPPED, `p` is
 * a pinned host allocation read through its device-mapped address over the
 * host link.  A measurement and verification helper: it gives the bandwidth
 * at which the SMs read HBM or host memory (the roofline of the host-weight
 * mode of the grouped GEMM) and lets tests compare buffer contents.
 */
bsf_status bsf_checksum_u64(const void* p, size_t bytes, int flags, unsigned long long* out, bsf_stream_t stream);

/* ------------------------------------------------------------------------
 * NVFP4 operands ("AsymGEMM" README, "FP4 Asymmetric GEMM": E2M1 data packed
 * two elements per byte, FP8 E4M3 scale factors; "CuTeDSL bei Perplexity":
 * one scale per 16 elements).  Formats:
 *   data   uint8 rows of K/2 bytes; element 2i in the low nibble of byte i;
 *          E2M1 = sign, 2 exponent bits (bias 1), 1 mantissa bit:
 *          0, 0.5, 1, 1.5, 2, 3, 4, 6.
 *   scales int32 words of four unsigned E4M3 bytes, byte i of word w for
 *          elements 64w + 16i .. 64w + 16i + 15 of its row; MN-major:
 *          activations [K/64][sf_ld] (sf_ld >= rows, multiple of 4),
 *          weights [E][K/64][N].
 *   tensor exponent j (int, |j| <= 100): a power-of-two scale 2**j of the
 *          whole activation tensor (a_exp) or of each expert's weights
 *          (b_exp, device int32 [E]); values outside are clamped.
 * value = e2m1 * scale * 2**j.  Quantisation of a block of 16: amax = max|x|,
 * scale = E4M3(amax / 6 * 2**-j) (nearest even, saturating at 448),
 * element = E2M1(x / (scale * 2**j)) (nearest even, saturating at 6), each
 * step one float32 operation rounded to nearest even; a zero scale stores
 * zero codes.
 */

/* bsf_nvfp4_tensor_exponent — for each of `groups` consecutive groups of
 * `per_group` bf16 values (per_group % 8 == 0): the least j with
 * max|x| <= 6 * 448 * 2**j (0 for an all-zero group), in [-100, 100], written
 * to exp_out (device int32 [groups]).  groups <= 65535. */
bsf_status bsf_nvfp4_tensor_exponent(const void* x, int64_t groups, int64_t per_group, int32_t* exp_out,
                                     bsf_stream_t stream);

/* bsf_quantise_act_nvfp4 — x bf16 [T, K] (K % 64 == 0) -> q uint8 [T, K/2],
 * sf int32 [K/64][sf_ld], with tensor exponent a_exp.  16-byte aligned x, q, sf. */
bsf_status bsf_quantise_act_nvfp4(const void* x, int64_t T, int64_t K, int a_exp, uint8_t* q, int32_t* sf,
                                  int64_t sf_ld, bsf_stream_t stream);

/* bsf_quantise_weight_nvfp4 — w bf16 [E, N, K] (K % 64 == 0) -> q uint8
 * [E, N, K/2], sfb int32 [E][K/64][N], expert e with exponent b_exp[e]
 * (device int32 [E], e.g. from bsf_nvfp4_tensor_exponent with per_group = N*K).
 * 1 x 16 blocks along K, like the activations. */
bsf_status bsf_quantise_weight_nvfp4(const void* w, int64_t E, int64_t N, int64_t K, const int32_t* b_exp,
                                     uint8_t* q, int32_t* sfb, bsf_stream_t stream);

/* bsf_dispatch_nvfp4 — bsf_dispatch for NVFP4 rows: quantise (tensor
 * exponent a_exp) + route + scatter in one launch for T*kr <=
 * BSF_DISPATCH_MAX_ASSIGNMENTS and E <= BSF_DISPATCH_MAX_EXPERTS.  a_packed
 * uint8 [m_cap, K/2], sfa_packed int32 [K/64][sfa_ld]; K % 64 == 0; the bytes
 * written equal bsf_quantise_act_nvfp4 followed by the row scatter.  Other
 * arguments, outputs and errors as in bsf_dispatch. */
bsf_status bsf_dispatch_nvfp4(const void* x, int64_t T, int64_t K, int a_exp, const int32_t* topk_ids, int64_t kr,
                              int64_t E, int layout, int64_t align_or_max_m, int32_t* counts, int32_t* seg_start,
                              int32_t* output_index, int32_t* token_of_row, int32_t* m_indices, int64_t m_cap,
                              uint8_t* a_packed, int32_t* sfa_packed, int64_t sfa_ld, bsf_stream_t stream);

/* bsf_route_nvfp4 — bsf_route whose scatter copies NVFP4 rows: q uint8 [T, K/2]
 * and sf int32 [K/64][sf_ld] (from bsf_quantise_act_nvfp4) into a_packed uint8
 * [m_cap, K/2] and sfa_packed int32 [K/64][sfa_ld]; K % 64 == 0.  Routing
 * outputs, workspace and errors as in bsf_route. */
bsf_status bsf_route_nvfp4(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout,
                           int64_t align_or_max_m, int32_t* counts, int32_t* seg_start, int32_t* output_index,
                           int32_t* token_of_row, int32_t* m_indices, int64_t m_cap, const uint8_t* q,
                           const int32_t* sf, int64_t sf_ld, int64_t K, uint8_t* a_packed, int32_t* sfa_packed,
                           int64_t sfa_ld, void* workspace, size_t workspace_bytes, bsf_stream_t stream);

/* bsf_grouped_gemm_nvfp4_contig / _masked — the grouped GEMMs of
 * bsf_grouped_gemm_contig / _masked on NVFP4 operands:
 *   D[r, n] = BF16( 2**(a_exp + b_exp[e]) * sum_k e2m1(A[r,k]) sA[r,k/16] e2m1(B_e[n,k]) sB_e[n,k/16] )
 * FP32 accumulation on the tensor cores (block-scaled MMA, kind::mxf4nvf4),
 * the power-of-two tensor scale applied exactly to the accumulator, then
 * round-to-nearest-even to bf16.  a uint8 [rows, K/2], b uint8 [E, N, K/2]
 * (device, or pinned host with BSF_B_HOST_MAPPED), sfa / sfb as above,
 * b_exp device int32 [E] or NULL (all 0).  Needs K % 256 == 0, N % 128 == 0,
 * E <= 256 (else BSF_ERR_UNSUPPORTED), 16-byte aligned a, b, d, sfa, sfb.
 * Rows, segments, masks, ownership, launch order and errors as in the FP8
 * calls. */
bsf_status bsf_grouped_gemm_nvfp4_contig(const uint8_t* a, const int32_t* sfa, int64_t sfa_ld, int64_t m_cap,
                                         int a_exp, const uint8_t* b, const int32_t* sfb, const int32_t* b_exp,
                                         void* d, const int32_t* seg_start, const int32_t* counts, int64_t E,
                                         int64_t N, int64_t K, int flags, bsf_stream_t stream);
bsf_status bsf_grouped_gemm_nvfp4_masked(const uint8_t* a, const int32_t* sfa, int64_t sfa_ld, int a_exp,
                                         const uint8_t* b, const int32_t* sfb, const int32_t* b_exp, void* d,
                                         const int32_t* masked_m, int64_t E, int64_t max_m, int64_t N, int64_t K,
                                         int64_t expected_m, int flags, bsf_stream_t stream);

/* ------------------------------------------------------------------------
 * BF16 operands ("AsymGEMM" README, "BF16 Asymmetric GEMM": a bf16 [M, K],
 * b bf16 [G, N, K], d bf16 [M, N]; contiguous and masked layouts as for FP8).
 */

/* bsf_route_bf16 — bsf_route whose scatter copies bf16 rows: x bf16 [T, K]
 * (K % 8 == 0) into a_packed bf16 [m_cap, K] (routed rows written, padding
 * rows left as they were).  Routing outputs, workspace and errors as in
 * bsf_route; x may be NULL (indices only). */
bsf_status bsf_route_bf16(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout,
                          int64_t align_or_max_m, int32_t* counts, int32_t* seg_start, int32_t* output_index,
                          int32_t* token_of_row, int32_t* m_indices, int64_t m_cap, const void* x, int64_t K,
                          void* a_packed, void* workspace, size_t workspace_bytes, bsf_stream_t stream);

/* bsf_grouped_gemm_bf16_contig / _masked — D[r, n] = BF16( sum_k A[r, k] B_e[n, k] )
 * for the rows of each expert (contiguous segments seg_start / counts, or
 * masked slots of max_m rows with masked_m valid): FP32 accumulation on the
 * tensor cores (kind::f16, both operands BF16), round-to-nearest-even to
 * bf16.  a bf16 [rows, K], b bf16 [E, N, K] (device, or pinned host with
 * BSF_B_HOST_MAPPED), d bf16 [rows, N] (only the rows above are written).
 * Needs K % 64 == 0, N % 128 == 0, 16-byte aligned a, b, d.  Ownership,
 * launch order and errors as in the FP8 calls. */
bsf_status bsf_grouped_gemm_bf16_contig(const void* a, int64_t m_cap, const void* b, void* d,
                                        const int32_t* seg_start, const int32_t* counts, int64_t E, int64_t N,
                                        int64_t K, int flags, bsf_stream_t stream);
bsf_status bsf_grouped_gemm_bf16_masked(const void* a, const void* b, void* d, const int32_t* masked_m, int64_t E,
                                        int64_t max_m, int64_t N, int64_t K, int64_t expected_m, int flags,
                                        bsf_stream_t stream);

/* ------------------------------------------------------------------------
 * FP8 E4M3 with float32 scale factors ("AsymGEMM" README, notation:
 * disable_ue8m0_cast keeps the scale factors in float32 rather than UE8M0).
 * Per block (1 x 128 along K for activations, 128 x 128 for weights):
 * s = amax / 448 (one float32 division, nearest even; 1 for an all-zero
 * block), q = E4M3(x / s) (one float32 division, nearest-even E4M3,
 * saturating).  Scales: activations float32 [K/128][sf_ld] (MN-major,
 * sf_ld >= rows, multiple of 4); weights float32 [E][N/128][K/128].
 */

/* bsf_quantise_act_f32sf — x bf16 [T, K] (K % 128 == 0) -> q e4m3 [T, K], sf float32 [K/128][sf_ld]. */
bsf_status bsf_quantise_act_f32sf(const void* x, int64_t T, int64_t K, uint8_t* q, float* sf, int64_t sf_ld,
                                  bsf_stream_t stream);

/* bsf_quantise_weight_f32sf — w bf16 [E, N, K] -> q e4m3 [E, N, K], sf float32 [E][N/128][K/128]. */
bsf_status bsf_quantise_weight_f32sf(const void* w, int64_t E, int64_t N, int64_t K, uint8_t* q, float* sf,
                                     bsf_stream_t stream);

/* bsf_route_f32sf — bsf_route whose scatter copies e4m3 rows with their
 * float32 scale columns (q [T, K], sf [K/128][sf_ld] -> a_packed [m_cap, K],
 * sfa_packed [K/128][sfa_ld]).  Everything else as in bsf_route. */
bsf_status bsf_route_f32sf(const int32_t* topk_ids, int64_t T, int64_t kr, int64_t E, int layout,
                           int64_t align_or_max_m, int32_t* counts, int32_t* seg_start, int32_t* output_index,
                           int32_t* token_of_row, int32_t* m_indices, int64_t m_cap, const uint8_t* q,
                           const float* sf, int64_t sf_ld, int64_t K, uint8_t* a_packed, float* sfa_packed,
                           int64_t sfa_ld, void* workspace, size_t workspace_bytes, bsf_stream_t stream);

/* bsf_grouped_gemm_f32sf_contig / _masked — D[r, n] = BF16( sum_kb sA[r, kb]
 * sB_e[n/128, kb] sum_{k in kb} A[r, k] B_e[n, k] ) over 128-wide K-blocks
 * kb: every block is an unscaled FP8 MMA into its own FP32 partial (tensor
 * memory), then scaled and added in FP32 in K-block order on the CUDA cores.
 * Tiles of up to 64 tokens with one CTA per SM, or, for masked calls with
 * max_m <= 32 or expected_m <= 16 (a hint; 0 = unknown), of up to 32 tokens
 * with two CTAs per SM; an expert with more rows is split into chunks, each
 * streaming the expert's weights.  Needs
 * N % 128 == 0, K % 128 == 0, 16-byte aligned a, b, d, sfa.  Segments,
 * masks, flags (BSF_B_HOST_MAPPED: b and sfb pinned host memory), launch
 * order and errors as in the UE8M0 calls. */
bsf_status bsf_grouped_gemm_f32sf_contig(const uint8_t* a, const float* sfa, int64_t sfa_ld, int64_t m_cap,
                                         const uint8_t* b, const float* sfb, void* d, const int32_t* seg_start,
                                         const int32_t* counts, int64_t E, int64_t N, int64_t K, int flags,
                                         bsf_stream_t stream);
bsf_status bsf_grouped_gemm_f32sf_masked(const uint8_t* a, const float* sfa, int64_t sfa_ld, const uint8_t* b,
                                         const float* sfb, void* d, const int32_t* masked_m, int64_t E,
                                         int64_t max_m, int64_t N, int64_t K, int64_t expected_m, int flags,
                                         bsf_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BSFROUTE_H */
