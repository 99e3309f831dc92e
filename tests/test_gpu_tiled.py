"""The tiled weight layout (BSF_B_TILED): the tiling kernel is a byte permutation
checked against numpy, and every grouped GEMM entry point gives bit-identical
output on tiled and row-major weights (the same MMAs on the same bytes; only
the address each 128 x 128-byte weight box is loaded from changes).  One case
per format is also checked against the oracle directly.
"""

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_route_gb300 import MoEPath, ops
from tests.gpu_util import bits16, check_expert_block, require_gpu, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _np_tiled(b):
    """Row-major [E, N, row_bytes] bytes -> [E][N/128][row_bytes/128][128][128]."""
    E, N, R = b.shape
    return b.reshape(E, N // 128, 128, R // 128, 128).transpose(0, 1, 3, 2, 4).reshape(E, N, R)


@pytest.mark.parametrize("E,N,R", [(1, 128, 128), (3, 256, 384), (2, 384, 1024)])
def test_tile_kernel_is_the_block_permutation(dev, E, N, R):
    g = torch.Generator().manual_seed(E * 1000 + R)
    b = torch.randint(0, 256, (E, N, R), generator=g, dtype=torch.uint8)
    t = ops.tile_weights(b.to(dev))
    torch.cuda.synchronize()
    assert np.array_equal(u8(t), _np_tiled(b.numpy()))


def test_tile_kernel_bf16_rows(dev):
    w = (torch.randn(2, 256, 320) * 0.1).to(torch.bfloat16)
    t = ops.tile_weights(w.to(dev))
    torch.cuda.synchronize()
    assert t.shape == (2, 256, 640)
    assert np.array_equal(u8(t), _np_tiled(w.view(torch.uint8).numpy().reshape(2, 256, 640)))


def _x(rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g) * torch.exp2(torch.randint(-4, 5, (rows, 1), generator=g).float())
    return x.to(torch.bfloat16)


def _w(E, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(E, N, K, generator=g) * 0.02).to(torch.bfloat16)


def _same(d0, d1, seg, counts, what):
    for e in range(len(counts)):
        s, c = int(seg[e]), int(counts[e])
        assert torch.equal(d0[s:s + c].view(torch.int16), d1[s:s + c].view(torch.int16)), f"{what} expert {e}"


CONTIG_COUNTS = np.array([1, 15, 16, 17, 0, 33, 255, 257, 600, 2])
MASKED_CASES = [(64, 0), (64, 8), (320, 0), (320, 16)]


def _seg(counts, align):
    return np.concatenate([[0], np.cumsum((counts + align - 1) // align * align)])


def _masked(max_m):
    return np.minimum(np.array([0, 1, 16, 63, 64, max_m // 2, max_m, 7]), max_m)


# ---- FP8 (UE8M0 scales) ---------------------------------------------------------------------------

def _fp8_ops(x, w, dev):
    aq, asf = ops.quantise_act(x.to(dev))
    bq, sf128 = ops.quantise_weight(w.to(dev))
    return aq, asf, bq, ops.prepare_weight_sf(sf128, w.shape[2])


@pytest.mark.parametrize("align", [1, 128])
def test_fp8_contig(dev, align):
    E, N, K = len(CONTIG_COUNTS), 256, 640
    seg = _seg(CONTIG_COUNTS, align)
    x, w = _x(int(seg[-1]), K, 1 + align), _w(E, N, K, 2 + align)
    aq, asf, bq, sfb = _fp8_ops(x, w, dev)
    segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
    ct = torch.as_tensor(CONTIG_COUNTS, dtype=torch.int32, device=dev)
    d0 = ops.grouped_gemm_contig(aq, asf, bq, sfb, segt, ct)
    d1 = ops.grouped_gemm_contig(aq, asf, ops.tile_weights(bq), sfb, segt, ct, flags=ops.B_TILED)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _same(d0, d1, seg, CONTIG_COUNTS, f"fp8 contig align={align}")
    if align == 1:
        aq_r, asf_r = oracle.quantise.quantise_act(bits16(x))
        bq_r, bsf_r = oracle.quantise.quantise_weight(bits16(w))
        ref, _ = oracle.gemm.grouped_gemm(aq_r, asf_r, bq_r, bsf_r, seg, CONTIG_COUNTS)
        dg = bits16(d1)
        for e, c in enumerate(CONTIG_COUNTS):
            s = int(seg[e])
            if c:
                check_expert_block(dg[s:s + c], ref[s:s + c], f"fp8 tiled expert {e}")


@pytest.mark.parametrize("max_m,expected_m", MASKED_CASES)
def test_fp8_masked(dev, max_m, expected_m):
    masked = _masked(max_m)
    E, N, K = len(masked), 384, 512
    x, w = _x(E * max_m, K, 3 + max_m), _w(E, N, K, 4 + max_m)
    aq, asf, bq, sfb = _fp8_ops(x, w, dev)
    mt = torch.as_tensor(masked, dtype=torch.int32, device=dev)
    d0 = ops.grouped_gemm_masked(aq, asf, bq, sfb, mt, max_m, expected_m=expected_m)
    d1 = ops.grouped_gemm_masked(aq, asf, ops.tile_weights(bq), sfb, mt, max_m, expected_m=expected_m,
                                 flags=ops.B_TILED)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _same(d0, d1, np.arange(E + 1) * max_m, masked, f"fp8 masked max_m={max_m} expected_m={expected_m}")


@pytest.mark.parametrize("layout", [ops.CONTIGUOUS, ops.MASKED])
def test_fp8_host_mapped_tiled(dev, layout):
    counts = np.array([5, 0, 300, 40]) if layout == ops.CONTIGUOUS else np.array([5, 0, 64, 40])
    E, N, K = len(counts), 256, 512
    max_m = 64
    seg = _seg(counts, 1) if layout == ops.CONTIGUOUS else np.arange(E + 1) * max_m
    x, w = _x(int(seg[-1]), K, 5), _w(E, N, K, 6)
    aq, asf, bq, sfb = _fp8_ops(x, w, dev)
    bt_host = ops.tile_weights(bq).cpu().pin_memory()
    sfb_host = sfb.cpu().pin_memory()
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    if layout == ops.CONTIGUOUS:
        segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
        d0 = ops.grouped_gemm_contig(aq, asf, bq, sfb, segt, ct)
        d1 = ops.grouped_gemm_contig(aq, asf, bt_host, sfb_host, segt, ct, flags=ops.B_TILED | ops.B_HOST_MAPPED)
    else:
        d0 = ops.grouped_gemm_masked(aq, asf, bq, sfb, ct, max_m)
        d1 = ops.grouped_gemm_masked(aq, asf, bt_host, sfb_host, ct, max_m, flags=ops.B_TILED | ops.B_HOST_MAPPED)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _same(d0, d1, seg, counts, f"fp8 host-mapped tiled layout={layout}")


# ---- NVFP4, BF16, FP32 scales -------------------------------------------------------------------

@pytest.mark.parametrize("layout,max_m,expected_m", [(ops.CONTIGUOUS, 0, 0), (ops.MASKED, 64, 0),
                                                     (ops.MASKED, 320, 16)])
def test_nvfp4(dev, layout, max_m, expected_m):
    counts = CONTIG_COUNTS if layout == ops.CONTIGUOUS else _masked(max_m)
    E, N, K = len(counts), 256, 512
    seg = _seg(counts, 1) if layout == ops.CONTIGUOUS else np.arange(E + 1) * max_m
    x, w = _x(int(seg[-1]), K, 7 + max_m), _w(E, N, K, 8 + max_m)
    aq, asf = ops.quantise_act_nvfp4(x.to(dev), 0)
    bq, sfb, b_exp = ops.quantise_weight_nvfp4(w.to(dev))
    bt = ops.tile_weights(bq)
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    if layout == ops.CONTIGUOUS:
        segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
        d0 = ops.grouped_gemm_nvfp4_contig(aq, asf, 0, bq, sfb, b_exp, segt, ct)
        d1 = ops.grouped_gemm_nvfp4_contig(aq, asf, 0, bt, sfb, b_exp, segt, ct, flags=ops.B_TILED)
    else:
        d0 = ops.grouped_gemm_nvfp4_masked(aq, asf, 0, bq, sfb, b_exp, ct, max_m, expected_m=expected_m)
        d1 = ops.grouped_gemm_nvfp4_masked(aq, asf, 0, bt, sfb, b_exp, ct, max_m, expected_m=expected_m,
                                           flags=ops.B_TILED)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _same(d0, d1, seg, counts, f"nvfp4 layout={layout} max_m={max_m}")


@pytest.mark.parametrize("layout,max_m,expected_m", [(ops.CONTIGUOUS, 0, 0), (ops.MASKED, 64, 0),
                                                     (ops.MASKED, 320, 16)])
def test_bf16(dev, layout, max_m, expected_m):
    counts = CONTIG_COUNTS if layout == ops.CONTIGUOUS else _masked(max_m)
    E, N, K = len(counts), 256, 576
    seg = _seg(counts, 1) if layout == ops.CONTIGUOUS else np.arange(E + 1) * max_m
    x, w = _x(int(seg[-1]), K, 9 + max_m), _w(E, N, K, 10 + max_m)
    xd, wd = x.to(dev), w.to(dev)
    wt = ops.tile_weights(wd)
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    if layout == ops.CONTIGUOUS:
        segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
        d0 = ops.grouped_gemm_bf16_contig(xd, wd, segt, ct)
        d1 = ops.grouped_gemm_bf16_contig(xd, wt, segt, ct, flags=ops.B_TILED)
    else:
        d0 = ops.grouped_gemm_bf16_masked(xd, wd, ct, max_m, expected_m=expected_m)
        d1 = ops.grouped_gemm_bf16_masked(xd, wt, ct, max_m, expected_m=expected_m, flags=ops.B_TILED)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _same(d0, d1, seg, counts, f"bf16 layout={layout} max_m={max_m}")
    if layout == ops.CONTIGUOUS:
        ref, _ = oracle.bf16.grouped_gemm(bits16(x), bits16(w), seg, counts)
        dg = bits16(d1)
        for e, c in enumerate(counts):
            s = int(seg[e])
            if c:
                check_expert_block(dg[s:s + c], ref[s:s + c], f"bf16 tiled expert {e}")


@pytest.mark.parametrize("layout,max_m,expected_m", [(ops.CONTIGUOUS, 0, 0), (ops.MASKED, 64, 8),
                                                     (ops.MASKED, 200, 0)])
def test_f32sf(dev, layout, max_m, expected_m):
    counts = CONTIG_COUNTS if layout == ops.CONTIGUOUS else _masked(max_m)
    E, N, K = len(counts), 256, 512
    seg = _seg(counts, 1) if layout == ops.CONTIGUOUS else np.arange(E + 1) * max_m
    x, w = _x(int(seg[-1]), K, 11 + max_m), _w(E, N, K, 12 + max_m)
    aq, asf = ops.quantise_act_f32sf(x.to(dev))
    bq, bsf = ops.quantise_weight_f32sf(w.to(dev))
    bt = ops.tile_weights(bq)
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    if layout == ops.CONTIGUOUS:
        segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
        d0 = ops.grouped_gemm_f32sf_contig(aq, asf, bq, bsf, segt, ct)
        d1 = ops.grouped_gemm_f32sf_contig(aq, asf, bt, bsf, segt, ct, flags=ops.B_TILED)
    else:
        d0 = ops.grouped_gemm_f32sf_masked(aq, asf, bq, bsf, ct, max_m, expected_m=expected_m)
        d1 = ops.grouped_gemm_f32sf_masked(aq, asf, bt, bsf, ct, max_m, expected_m=expected_m, flags=ops.B_TILED)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _same(d0, d1, seg, counts, f"f32sf layout={layout} max_m={max_m}")


# ---- the whole path --------------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["fp8", "nvfp4", "bf16", "fp8_f32sf"])
@pytest.mark.parametrize("layout", [ops.CONTIGUOUS, ops.MASKED])
def test_moe_path_tiled_equals_row_major(dev, fmt, layout):
    E, kr, T, K, N = 16, 4, 96, 512, 256
    g = torch.Generator().manual_seed(13)
    x = _x(T, K, 14)
    w = _w(E, N, K, 15)
    ids = torch.stack([torch.randperm(E, generator=g)[:kr] for _ in range(T)]).to(torch.int32)
    p = torch.rand(T, kr, generator=g)
    a_or_m = 128 if layout == ops.CONTIGUOUS else 64
    out = []
    for tiled in (False, True):
        path = MoEPath(E, kr, T, K, N, w, layout=layout, align_or_max_m=a_or_m, device=dev, fmt=fmt,
                       expected_m=T * kr // E, tiled_weights=tiled)
        out.append(path.step(x.to(dev), ids.to(dev), p.to(dev)).clone())
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    assert torch.equal(out[0].view(torch.int16), out[1].view(torch.int16))
