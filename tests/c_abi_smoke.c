/*
 * A plain C caller of libbsfroute: the whole FP8 path through the C ABI of
 * include/bsfroute.h alone (no Python, no PyTorch), on buffers from cudaMalloc.
 *
 *   c_abi_smoke DIR T KR E K N ALIGN
 *
 * reads DIR/x.bin (bf16 [T, K]), DIR/w.bin (bf16 [E, N, K]), DIR/ids.bin
 * (int32 [T, KR]) and DIR/p.bin (fp32 [T, KR]); runs
 *   bsf_quantise_weight -> bsf_prepare_weight_sf -> bsf_tile_weights (once)
 *   bsf_quantise_act -> bsf_route (+ scatter) -> bsf_grouped_gemm_contig -> bsf_combine
 * on one stream, and writes the combined output to DIR/z.bin (bf16 [T, N]) and
 * the packed-row index to DIR/output_index.bin (int32 [T, KR]).  Exits non-zero
 * with a message on any failed call or a non-zero device error word.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "bsfroute.h"

static int fail(const char* what, const char* why) {
  fprintf(stderr, "c_abi_smoke: %s: %s\n", what, why);
  return 1;
}

#define CUDA(call)                                                          \
  do {                                                                      \
    cudaError_t e_ = (call);                                                \
    if (e_ != cudaSuccess) return fail(#call, cudaGetErrorString(e_));      \
  } while (0)
#define BSF(call)                                                           \
  do {                                                                      \
    bsf_status s_ = (call);                                                 \
    if (s_ != BSF_OK) return fail(#call, bsf_status_string(s_));            \
  } while (0)

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* buf = malloc(bytes ? bytes : 1);
  const size_t got = buf ? fread(buf, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(buf);
    return NULL;
  }
  return buf;
}

static int write_file(const char* dir, const char* name, const void* data, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  const size_t put = fwrite(data, 1, bytes, f);
  fclose(f);
  return put != bytes;
}

static int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

int main(int argc, char** argv) {
  if (argc != 8) return fail("usage", "c_abi_smoke DIR T KR E K N ALIGN");
  const char* dir = argv[1];
  const int64_t T = atoll(argv[2]), kr = atoll(argv[3]), E = atoll(argv[4]), K = atoll(argv[5]), N = atoll(argv[6]),
                align = atoll(argv[7]);
  if (T <= 0 || kr <= 0 || E <= 0 || K <= 0 || N <= 0 || align <= 0) return fail("arguments", "sizes must be > 0");

  uint16_t* hx = read_file(dir, "x.bin", (size_t)(T * K * 2));
  uint16_t* hw = read_file(dir, "w.bin", (size_t)(E * N * K * 2));
  int32_t* hids = read_file(dir, "ids.bin", (size_t)(T * kr * 4));
  float* hp = read_file(dir, "p.bin", (size_t)(T * kr * 4));
  if (!hx || !hw || !hids || !hp) return fail("inputs", "missing or short input file");

  /* sizes from the header's contracts: m_cap = T*kr + E*(align-1); SF words per row ceil(K/512);
     packed SF leading dimension rows rounded up to 4 */
  const int64_t m_cap = T * kr + E * (align - 1);
  const int64_t nw = (K + 511) / 512;
  const int64_t sf_ld_t = round_up(T, 4), sf_ld_m = round_up(m_cap, 4);
  const size_t ws_bytes = bsf_route_workspace_bytes(T, kr, E);

  cudaStream_t s;
  CUDA(cudaStreamCreate(&s));
  void *dx, *dw, *dz, *dy, *dws;
  uint8_t *dwq, *dwt, *dq, *da;
  float *dsf128, *dp;
  int32_t *dsfb, *dsf, *dsfa, *dids, *dcounts, *dseg, *doi, *dtok;
  CUDA(cudaMalloc(&dx, T * K * 2));
  CUDA(cudaMalloc(&dw, E * N * K * 2));
  CUDA(cudaMalloc((void**)&dwq, E * N * K));
  CUDA(cudaMalloc((void**)&dwt, E * N * K));
  CUDA(cudaMalloc((void**)&dsf128, E * (N / 128) * (K / 128) * 4));
  CUDA(cudaMalloc((void**)&dsfb, E * nw * N * 4));
  CUDA(cudaMalloc((void**)&dq, T * K));
  CUDA(cudaMalloc((void**)&dsf, nw * sf_ld_t * 4));
  CUDA(cudaMalloc((void**)&dids, T * kr * 4));
  CUDA(cudaMalloc((void**)&dp, T * kr * 4));
  CUDA(cudaMalloc((void**)&dcounts, E * 4));
  CUDA(cudaMalloc((void**)&dseg, (E + 1) * 4));
  CUDA(cudaMalloc((void**)&doi, T * kr * 4));
  CUDA(cudaMalloc((void**)&dtok, m_cap * 4));
  CUDA(cudaMalloc((void**)&da, m_cap * K));
  CUDA(cudaMalloc((void**)&dsfa, nw * sf_ld_m * 4));
  CUDA(cudaMalloc(&dws, ws_bytes ? ws_bytes : 16));
  CUDA(cudaMalloc(&dy, m_cap * N * 2));
  CUDA(cudaMalloc(&dz, T * N * 2));

  CUDA(cudaMemcpyAsync(dx, hx, T * K * 2, cudaMemcpyHostToDevice, s));
  CUDA(cudaMemcpyAsync(dw, hw, E * N * K * 2, cudaMemcpyHostToDevice, s));
  CUDA(cudaMemcpyAsync(dids, hids, T * kr * 4, cudaMemcpyHostToDevice, s));
  CUDA(cudaMemcpyAsync(dp, hp, T * kr * 4, cudaMemcpyHostToDevice, s));

  /* once per weight load */
  BSF(bsf_quantise_weight(dw, E, N, K, dwq, dsf128, s));
  BSF(bsf_prepare_weight_sf(dsf128, E, N, K, dsfb, s));
  BSF(bsf_tile_weights(dwq, E, N, K, dwt, s));
  /* the step */
  BSF(bsf_quantise_act(dx, T, K, dq, dsf, sf_ld_t, s));
  BSF(bsf_route(dids, T, kr, E, BSF_LAYOUT_CONTIGUOUS, align, dcounts, dseg, doi, dtok, NULL, m_cap, dq, dsf,
                sf_ld_t, K, da, dsfa, sf_ld_m, dws, ws_bytes, s));
  BSF(bsf_grouped_gemm_contig(da, dsfa, sf_ld_m, m_cap, dwt, dsfb, dy, dseg, dcounts, E, N, K, BSF_B_TILED, s));
  BSF(bsf_combine(dy, m_cap, doi, dp, T, kr, N, dz, s));

  uint16_t* hz = malloc((size_t)(T * N * 2));
  int32_t* hoi = malloc((size_t)(T * kr * 4));
  if (!hz || !hoi) return fail("malloc", "out of host memory");
  CUDA(cudaMemcpyAsync(hz, dz, T * N * 2, cudaMemcpyDeviceToHost, s));
  CUDA(cudaMemcpyAsync(hoi, doi, T * kr * 4, cudaMemcpyDeviceToHost, s));
  CUDA(cudaStreamSynchronize(s));
  int32_t derr = 0;
  BSF(bsf_get_device_error(&derr, 1, s));
  if (derr != 0) return fail("device error word", "non-zero");
  if (write_file(dir, "z.bin", hz, (size_t)(T * N * 2)) || write_file(dir, "output_index.bin", hoi, (size_t)(T * kr * 4)))
    return fail("outputs", "cannot write");

  cudaFree(dx); cudaFree(dw); cudaFree(dwq); cudaFree(dwt); cudaFree(dsf128); cudaFree(dsfb); cudaFree(dq);
  cudaFree(dsf); cudaFree(dids); cudaFree(dp); cudaFree(dcounts); cudaFree(dseg); cudaFree(doi); cudaFree(dtok);
  cudaFree(da); cudaFree(dsfa); cudaFree(dws); cudaFree(dy); cudaFree(dz);
  CUDA(cudaStreamDestroy(s));
  free(hx); free(hw); free(hids); free(hp); free(hz); free(hoi);
  printf("c_abi_smoke ok\n");
  return 0;
}
