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
