"""CPU-side checks of the C-ABI library: it builds, loads, and exports every
symbol that include/bsfroute.h declares (no compute calls: no GPU here)."""

import ctypes

import pytest

from block_scaled_fp8_route_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    path = build.build()
    return _lib.load(path)


def test_every_header_symbol_is_exported(lib):
    names = _lib.header_symbols()
    assert "bsf_grouped_gemm_contig" in names and "bsf_route" in names
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(_lib.SIGNATURES), "binding signatures out of sync with the header"


def test_host_only_calls(lib):
    assert lib.bsf_version() >= 1
    assert lib.bsf_status_string(0) == b"ok"
    assert lib.bsf_status_string(2).startswith(b"pointer")
    # workspace size is host arithmetic: one int32 per (chunk, expert), the chunk the smallest of
    # 512 / 1024 / 2048 assignments that keeps the batch within 64 chunks (else 2048)
    assert lib.bsf_route_workspace_bytes(4096, 8, 128) == 64 * 128 * 4       # 32768 / 512
    assert lib.bsf_route_workspace_bytes(8192, 8, 256) == 64 * 256 * 4       # 65536 / 1024
    assert lib.bsf_route_workspace_bytes(8193, 8, 256) == 33 * 256 * 4       # 65544 -> 2048-chunks
    assert lib.bsf_route_workspace_bytes(65536, 8, 16) == 256 * 16 * 4       # 524288 / 2048 (route_scan)
    assert lib.bsf_route_workspace_bytes(1, 1, 4) == 16
    # T * kr above INT32_MAX: refused (0 bytes) without forming the product
    assert lib.bsf_route_workspace_bytes(2**31, 8, 8) == 0
    assert lib.bsf_route_workspace_bytes(2**62, 4, 8) == 0


def test_argument_validation_needs_no_device(lib):
    nul = ctypes.c_void_p(0)
    # K not a multiple of 128 is rejected before anything touches the device
    assert lib.bsf_quantise_act(nul, 4, 100, nul, nul, 4, nul) == 1
    # N not a multiple of 128
    assert lib.bsf_grouped_gemm_contig(nul, nul, 4, 4, nul, nul, nul, nul, nul, 2, 100, 128, 0, nul) == 1
    # unknown layout
    assert lib.bsf_route(nul, 4, 2, 4, 7, 1, nul, nul, nul, nul, nul, 8, nul, nul, 0, 0, nul, nul, 0, nul, 0,
                         nul) == 1
    # T * kr above INT32_MAX (would wrap as a 64-bit product too at T = 2**62): unsupported, nothing enqueued
    fake = ctypes.c_void_p(256)
    for T, kr in ((2**31, 8), (2**62, 4)):
        assert lib.bsf_route(nul, T, kr, 8, 0, 1, fake, fake, fake, fake, nul, 1 << 30, nul, nul, 0, 0, nul, nul, 0,
                             fake, 1 << 20, nul) == 3
        assert lib.bsf_route_no_alloc(nul, T, kr, 8, 0, 1, fake, fake, fake, fake, nul, 1 << 30, nul, nul, 0, 0, nul,
                                      nul, 0, nul) == 3
    # row-filtered quantiser: the row filter is required
    assert lib.bsf_quantise_act_rows(fake, 4, 128, nul, fake, fake, fake, 4, nul) == 1
    # fused route + quantise: K a multiple of 128, at most 32 routes per token, 16-byte aligned buffers
    odd = ctypes.c_void_p(264)
    assert lib.bsf_route_quantise(fake, 4, 100, nul, 2, 4, 0, 1, fake, fake, fake, fake, nul, 8, fake, fake, 8,
                                  fake, 64, nul) == 1
    assert lib.bsf_route_quantise(fake, 4, 128, nul, 33, 4, 0, 1, fake, fake, fake, fake, nul, 200, fake, fake, 200,
                                  fake, 64, nul) == 3
    assert lib.bsf_route_quantise(odd, 4, 128, nul, 2, 4, 0, 1, fake, fake, fake, fake, nul, 8, fake, fake, 8,
                                  fake, 64, nul) == 2
    # combine with N not a multiple of 8
    assert lib.bsf_combine(nul, 4, nul, nul, 2, 2, 12, nul, nul) == 1
    # dispatch: batch above the single-launch limit is unsupported, K not a multiple of 128 invalid
    assert lib.bsf_dispatch(nul, 4096, 128, nul, 8, 128, 0, 1, nul, nul, nul, nul, nul, 1 << 20, nul, nul, 1 << 20,
                            nul) == 3
    assert lib.bsf_dispatch(nul, 4, 100, nul, 2, 4, 0, 1, nul, nul, nul, nul, nul, 8, nul, nul, 8, nul) == 1
    # NVFP4: K must be a multiple of 256 for the GEMM, of 64 for the quantiser; tensor exponent within +-100
    assert lib.bsf_grouped_gemm_nvfp4_masked(nul, nul, 64, 0, nul, nul, nul, nul, nul, 2, 32, 128, 128, 0, 0,
                                             nul) == 1
    assert lib.bsf_quantise_act_nvfp4(nul, 4, 96, 0, nul, nul, 4, nul) == 1
    assert lib.bsf_quantise_act_nvfp4(nul, 4, 128, 101, nul, nul, 4, nul) == 1
    assert lib.bsf_grouped_gemm_nvfp4_contig(nul, nul, 8, 8, 0, nul, nul, nul, nul, nul, nul, 300, 128, 256, 0,
                                             nul) == 3                      # more than 256 experts
    # BF16: K must be a multiple of 64
    assert lib.bsf_grouped_gemm_bf16_contig(nul, 8, nul, nul, nul, nul, 2, 128, 96, 0, nul) == 1
    # FP32 scales: N must be a multiple of 128
    assert lib.bsf_grouped_gemm_f32sf_masked(nul, nul, 8, nul, nul, nul, nul, 2, 4, 100, 128, 0, 0, nul) == 1
    # weight tiling: rows of a multiple of 128 bytes, N a multiple of 128, distinct buffers
    assert lib.bsf_tile_weights(nul, 2, 128, 96, nul, nul) == 1
    assert lib.bsf_tile_weights(nul, 2, 100, 128, nul, nul) == 1
    assert lib.bsf_tile_weights(nul, 2, 128, 128, nul, nul) == 1
    # an undefined GEMM flag bit
    assert lib.bsf_grouped_gemm_contig(nul, nul, 4, 4, nul, nul, nul, nul, nul, 2, 128, 128, 0x4, nul) == 1


def test_python_constants_match_header():
    import os
    import re

    from block_scaled_fp8_route_gb300 import ops
    with open(os.path.join(build.ROOT, "include", "bsfroute.h")) as f:
        text = f.read()
    defs = {m.group(1): int(m.group(2), 0) for m in re.finditer(r"#define BSF_(\w+) (0x[0-9a-fA-F]+|\d+)", text)}
    for name in ("DEVERR_EXPERT_ID", "DEVERR_MASKED_OVERFLOW", "DEVERR_TIMEOUT", "DEVERR_BAD_SCALE",
                 "DEVERR_SEGMENT"):
        assert getattr(ops, name) == defs[name], name
    assert ops.B_HOST_MAPPED == defs["B_HOST_MAPPED"]
    assert ops.B_TILED == defs["B_TILED"]
    assert ops.DISPATCH_MAX_ASSIGNMENTS == defs["DISPATCH_MAX_ASSIGNMENTS"]
    assert ops.DISPATCH_MAX_EXPERTS == defs["DISPATCH_MAX_EXPERTS"]


def test_argument_validation_of_the_other_entry_points(lib):
    """Every entry point's host-side checks return their documented status before anything touches
    the device (the pointers below are never dereferenced: each call fails a check first)."""
    nul = ctypes.c_void_p(0)
    ok = ctypes.c_void_p(256)        # 16-byte aligned, never dereferenced
    odd = ctypes.c_void_p(264)       # not 16-byte aligned
    INVALID, MISALIGNED, UNSUPPORTED = 1, 2, 3
    big = 1 << 40

    # FP8 masked GEMM: a, sfa, sfa_ld, b, sfb, d, masked_m, E, max_m, N, K, expected_m, flags, stream
    def masked(a=ok, sfa=ok, sfa_ld=64, d=ok, masked_m=ok, E=2, max_m=32, N=128, K=128, flags=0):
        return lib.bsf_grouped_gemm_masked(a, sfa, sfa_ld, ok, ok, d, masked_m, E, max_m, N, K, 0, flags, nul)
    assert masked(max_m=0) == INVALID
    assert masked(N=100) == INVALID
    assert masked(K=64) == INVALID
    assert masked(E=1025) == INVALID                      # above the expert-table limit
    assert masked(flags=0x40) == INVALID                  # undefined flag bit
    assert masked(a=nul) == INVALID
    assert masked(sfa_ld=60) == INVALID                   # below E * max_m rows
    assert masked(sfa_ld=66) == INVALID                   # not a multiple of 4
    assert masked(d=odd) == MISALIGNED
    assert masked(masked_m=nul) == INVALID
    assert masked(E=1024, max_m=1 << 22, sfa_ld=1 << 32) == UNSUPPORTED   # E * max_m rows above INT32_MAX

    # FP32-scale contiguous GEMM: a, sfa, sfa_ld, m_cap, b, sfb, d, seg_start, counts, E, N, K, flags, stream
    def f32c(m_cap=64, K=128, seg=ok, sfa=ok):
        return lib.bsf_grouped_gemm_f32sf_contig(ok, sfa, 64, m_cap, ok, ok, ok, seg, ok, 2, 128, K, 0, nul)
    assert f32c(m_cap=-1) == INVALID
    assert f32c(m_cap=0) == 0                             # nothing to do
    assert f32c(K=96) == INVALID
    assert f32c(seg=nul) == INVALID
    assert f32c(sfa=odd) == MISALIGNED

    # BF16 masked GEMM: a, b, d, masked_m, E, max_m, N, K, expected_m, flags, stream
    def bf16m(max_m=32, K=128, masked_m=ok, b=ok):
        return lib.bsf_grouped_gemm_bf16_masked(ok, b, ok, masked_m, 2, max_m, 128, K, 0, 0, nul)
    assert bf16m(max_m=0) == INVALID
    assert bf16m(K=96) == INVALID
    assert bf16m(masked_m=nul) == INVALID
    assert bf16m(b=odd) == MISALIGNED

    # weight quantisers and the scale-factor transform: (w, E, N, K, q, sf, stream)
    for fn in (lib.bsf_quantise_weight, lib.bsf_quantise_weight_f32sf):
        assert fn(ok, 2, 128, 96, ok, ok, nul) == INVALID
        assert fn(ok, -1, 128, 128, ok, ok, nul) == INVALID
        assert fn(nul, 0, 128, 128, nul, nul, nul) == 0   # no experts: nothing to do
        assert fn(ok, 2, 128, 128, nul, ok, nul) == INVALID
        assert fn(odd, 2, 128, 128, ok, ok, nul) == MISALIGNED
    assert lib.bsf_prepare_weight_sf(ok, 2, 100, 128, ok, nul) == INVALID
    assert lib.bsf_prepare_weight_sf(nul, 0, 128, 128, nul, nul) == 0
    assert lib.bsf_prepare_weight_sf(nul, 2, 128, 128, ok, nul) == INVALID
    # NVFP4 weights: (w, E, N, K, b_exp, q, sfb, stream)
    assert lib.bsf_quantise_weight_nvfp4(ok, 0, 128, 128, ok, ok, ok, nul) == INVALID
    assert lib.bsf_quantise_weight_nvfp4(ok, 2, 128, 96, ok, ok, ok, nul) == INVALID
    assert lib.bsf_quantise_weight_nvfp4(ok, 2, 128, 128, nul, ok, ok, nul) == INVALID
    assert lib.bsf_quantise_weight_nvfp4(ok, 2, 128, 128, ok, ok, odd, nul) == MISALIGNED

    # FP32-scale activation quantiser: (x, T, K, q, sf, sf_ld, stream)
    assert lib.bsf_quantise_act_f32sf(ok, 4, 96, ok, ok, 4, nul) == INVALID
    assert lib.bsf_quantise_act_f32sf(ok, 8, 128, ok, ok, 4, nul) == INVALID      # sf_ld below T
    assert lib.bsf_quantise_act_f32sf(ok, 4, 128, ok, ok, 6, nul) == INVALID      # sf_ld not a multiple of 4
    assert lib.bsf_quantise_act_f32sf(nul, 0, 128, nul, nul, 0, nul) == 0
    assert lib.bsf_quantise_act_f32sf(ok, 4, 128, ok, odd, 4, nul) == MISALIGNED

    # routing with a scatter in the other formats: (ids, T, kr, E, layout, a_or_m, counts, seg_start,
    # output_index, token_of_row, m_indices, m_cap, q, sf, sf_ld, K, a_packed, sfa_packed, sfa_ld, ws, ws_bytes, s)
    def route(fn, T=4, kr=2, layout=0, K=128, q=ok, a_packed=ok):
        return fn(ok, T, kr, 4, layout, 1, ok, ok, ok, ok, nul, 64, q, ok, 8, K, a_packed, ok, 64, ok, big, nul)
    for fn, k_bad in ((lib.bsf_route_nvfp4, 96), (lib.bsf_route_f32sf, 64)):
        assert route(fn, layout=7) == INVALID
        assert route(fn, T=2**62, kr=4) == UNSUPPORTED
        assert route(fn, K=k_bad) == INVALID
        assert route(fn, q=odd) == MISALIGNED
    # BF16 rows: (ids, T, kr, E, layout, a_or_m, counts, seg_start, output_index, token_of_row, m_indices, m_cap,
    # x, K, a_packed, ws, ws_bytes, s)
    def route_bf16(T=4, kr=2, K=128, x=ok, a_packed=ok):
        return lib.bsf_route_bf16(ok, T, kr, 4, 0, 1, ok, ok, ok, ok, nul, 64, x, K, a_packed, ok, big, nul)
    assert route_bf16(T=2**62, kr=4) == UNSUPPORTED
    assert route_bf16(K=12) == INVALID                   # row bytes not a multiple of 16
    assert route_bf16(a_packed=nul) == INVALID
    assert route_bf16(x=odd) == MISALIGNED

    # NVFP4 single-launch dispatch: (x, T, K, a_exp, ids, kr, E, layout, a_or_m, counts, seg_start,
    # output_index, token_of_row, m_indices, m_cap, a_packed, sfa_packed, sfa_ld, s)
    def disp(T=4, K=128, a_exp=0, kr=2):
        return lib.bsf_dispatch_nvfp4(ok, T, K, a_exp, ok, kr, 4, 0, 1, ok, ok, ok, ok, nul, 64, ok, ok, 64, nul)
    assert disp(K=96) == INVALID
    assert disp(a_exp=101) == INVALID
    assert disp(T=4096, kr=8) == UNSUPPORTED             # above the single-launch limit
    assert disp(T=2**62, kr=4) == UNSUPPORTED            # T * kr would wrap
    assert lib.bsf_dispatch(ok, 2**62, 128, ok, 4, 4, 0, 1, ok, ok, ok, ok, nul, 64, ok, ok, 64, nul) == UNSUPPORTED

    # NVFP4 tensor exponent: (x, groups, per_group, exp_out, stream)
    assert lib.bsf_nvfp4_tensor_exponent(ok, 2, 12, ok, nul) == INVALID
    assert lib.bsf_nvfp4_tensor_exponent(ok, 2, 16, nul, nul) == INVALID
    assert lib.bsf_nvfp4_tensor_exponent(odd, 2, 16, ok, nul) == MISALIGNED
    assert lib.bsf_nvfp4_tensor_exponent(ok, 65536, 16, ok, nul) == UNSUPPORTED

    # checksum: (p, bytes, flags, out, stream)
    assert lib.bsf_checksum_u64(ok, 24, 0, ok, nul) == INVALID
    assert lib.bsf_checksum_u64(ok, 32, 0x2, ok, nul) == INVALID
    assert lib.bsf_checksum_u64(ok, 32, 0, nul, nul) == INVALID
    assert lib.bsf_checksum_u64(odd, 32, 0, ok, nul) == MISALIGNED


def test_sizes_beyond_any_real_problem_are_refused_before_they_can_wrap(lib):
    """Row counts above 2^31 - 1 or row widths above 2^24 return BSF_ERR_UNSUPPORTED before any product
    of them is formed (T = 2^62 with K = 2^20 would wrap a 64-bit grid computation)."""
    ok = ctypes.c_void_p(256)
    nul = ctypes.c_void_p(0)
    UNSUPPORTED = 3
    T, K = 2**62, 2**20
    assert lib.bsf_quantise_act(ok, T, K, ok, ok, T, nul) == UNSUPPORTED
    assert lib.bsf_quantise_act_rows(ok, T, K, ok, ok, ok, ok, T, nul) == UNSUPPORTED
    assert lib.bsf_quantise_act_f32sf(ok, T, K, ok, ok, T, nul) == UNSUPPORTED
    assert lib.bsf_quantise_act_nvfp4(ok, T, K, 0, ok, ok, T, nul) == UNSUPPORTED
    assert lib.bsf_quantise_act(ok, 64, 2**25, ok, ok, 64, nul) == UNSUPPORTED        # row wider than 2^24
    assert lib.bsf_combine(ok, 8, ok, ok, T, 2, 1024, ok, nul) == UNSUPPORTED
    assert lib.bsf_route_quantise(ok, T, K, ok, 1, 4, 0, 1, ok, ok, ok, ok, nul, 2**62, ok, ok, 2**62, ok, 64,
                                  nul) == UNSUPPORTED
    for E, N in ((2**40, 2**20), (2, 2**40)):
        assert lib.bsf_quantise_weight(ok, E, N, 128, ok, ok, nul) == UNSUPPORTED
        assert lib.bsf_quantise_weight_f32sf(ok, E, N, 128, ok, ok, nul) == UNSUPPORTED
        assert lib.bsf_prepare_weight_sf(ok, E, N, 128, ok, nul) == UNSUPPORTED
        assert lib.bsf_quantise_weight_nvfp4(ok, E, N, 128, ok, ok, ok, nul) == UNSUPPORTED
        assert lib.bsf_tile_weights(ok, E, N, 128, ctypes.c_void_p(512), nul) == UNSUPPORTED
