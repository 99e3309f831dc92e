"""GPU parity of the grouped GEMM against the float64 oracle.

Tolerance (per expert, over its valid rows): calc_diff <= 1e-3 and
|d - ref| <= 2**-7 |ref| + 1e-3 rms(ref), ref the oracle's bf16 output.
Covers ragged segments (1, 15, 16, 17, 31, 33, 255, 256, 257, 600 rows), empty
experts, a partial last SF word (K = 640), K = 128, both layouts, the
workloads' full sizes (sampled experts for the large ones), and bitwise
determinism over 20 runs.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from block_scaled_fp8_route_gb300 import ops
from tests.gpu_util import bits16, check_expert_block, i32, require_gpu, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _operands(rows, E, N, K, seed, dev):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(rows, K, generator=g) * torch.exp2(torch.randint(-4, 5, (rows, 1), generator=g).float()))
    x = x.to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g) * 0.02).to(torch.bfloat16)
    aq, asf = ops.quantise_act(x.to(dev))
    bq, sf128 = ops.quantise_weight(w.to(dev))
    sfb = ops.prepare_weight_sf(sf128, K)
    aq_ref, asf_ref = oracle.quantise.quantise_act(bits16(x))
    bq_ref, bsf_ref = oracle.quantise.quantise_weight(bits16(w))
    return (aq, asf, bq, sfb), (aq_ref, asf_ref, bq_ref, bsf_ref)


def _check_all(d, ref_ops, seg, counts, what):
    aq_ref, asf_ref, bq_ref, bsf_ref = ref_ops
    ref, valid = oracle.gemm.grouped_gemm(aq_ref, asf_ref, bq_ref, bsf_ref, seg, counts)
    dg = bits16(d)
    for e in range(len(counts)):
        c = int(counts[e])
        if c == 0:
            continue
        s = int(seg[e])
        check_expert_block(dg[s:s + c], ref[s:s + c], f"{what} expert {e} ({c} rows)")


@pytest.mark.parametrize("K", [128, 640, 1024])
@pytest.mark.parametrize("align", [1, 128])
def test_contig_ragged_segments(dev, K, align):
    counts = np.array([1, 15, 16, 17, 31, 33, 0, 255, 256, 257, 600, 2])
    E, N = len(counts), 256
    seg = np.concatenate([[0], np.cumsum((counts + align - 1) // align * align)])
    rows = int(seg[-1])
    (aq, asf, bq, sfb), ref_ops = _operands(rows, E, N, K, 10 + K + align, dev)
    d = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_contig(aq, asf, bq, sfb, torch.as_tensor(seg, dtype=torch.int32, device=dev),
                            torch.as_tensor(counts, dtype=torch.int32, device=dev), d=d)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check_all(d, ref_ops, seg, counts, f"contig K={K} align={align}")
    # rows outside the segments' valid parts are never written
    dv = d.float().cpu().numpy()
    for e in range(E):
        assert np.isnan(dv[seg[e] + counts[e]:seg[e + 1]]).all()


@pytest.mark.parametrize("max_m,expected_m,N", [(64, 0, 384), (320, 0, 384), (320, 16, 384), (320, 0, 512),
                                                 (128, 0, 512)])
def test_masked_ragged(dev, max_m, expected_m, N):
    """N = 384: 128-row weight tiles; N = 512: 256-row work items (two weight tiles per token chunk)."""
    masked = np.array([0, 1, 16, 63, 64, max_m // 2, max_m, 7])
    masked = np.minimum(masked, max_m)
    E, K = len(masked), 512
    (aq, asf, bq, sfb), ref_ops = _operands(E * max_m, E, N, K, max_m + expected_m, dev)
    d = torch.full((E * max_m, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_masked(aq, asf, bq, sfb, torch.as_tensor(masked, dtype=torch.int32, device=dev), max_m,
                            d=d, expected_m=expected_m)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    seg = np.arange(E + 1) * max_m
    _check_all(d, ref_ops, seg, masked, f"masked max_m={max_m}")


def test_masked_many_experts_small_slots(dev):
    """More than 256 experts with small slots: the small-batch tile with its 1024-expert tables."""
    rng = np.random.default_rng(5)
    E, N, K, max_m = 260, 128, 128, 32
    masked = rng.integers(0, max_m + 1, E)
    masked[:7] = 0
    (aq, asf, bq, sfb), ref_ops = _operands(E * max_m, E, N, K, 77, dev)
    d = torch.full((E * max_m, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_masked(aq, asf, bq, sfb, torch.as_tensor(masked, dtype=torch.int32, device=dev), max_m, d=d)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check_all(d, ref_ops, np.arange(E + 1) * max_m, masked, "masked E=260")


def test_contig_many_experts_wide_items(dev):
    """More than 256 experts with 256-row work items (the 1024-expert tile tables)."""
    rng = np.random.default_rng(12)
    E, N, K = 260, 256, 256
    counts = rng.integers(0, 40, E)
    counts[::7] = 0
    seg = np.concatenate([[0], np.cumsum(counts)])
    (aq, asf, bq, sfb), ref_ops = _operands(int(seg[-1]), E, N, K, 78, dev)
    d = torch.full((int(seg[-1]), N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_contig(aq, asf, bq, sfb, torch.as_tensor(seg, dtype=torch.int32, device=dev),
                            torch.as_tensor(counts, dtype=torch.int32, device=dev), d=d)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check_all(d, ref_ops, seg, counts, "contig E=260 wide items")


def test_grouped_equals_single_launches_bitwise(dev):
    counts = np.array([40, 0, 130, 7])
    E, N, K = 4, 256, 512
    seg = np.concatenate([[0], np.cumsum(counts)])
    (aq, asf, bq, sfb), _ = _operands(int(seg[-1]), E, N, K, 77, dev)
    d = ops.grouped_gemm_contig(aq, asf, bq, sfb, torch.as_tensor(seg, dtype=torch.int32, device=dev),
                                torch.as_tensor(counts, dtype=torch.int32, device=dev))
    for e in range(E):
        if counts[e] == 0:
            continue
        one = np.zeros(E, dtype=np.int32)
        one[e] = counts[e]
        d1 = ops.grouped_gemm_contig(aq, asf, bq, sfb, torch.as_tensor(seg, dtype=torch.int32, device=dev),
                                     torch.as_tensor(one, device=dev))
        s, c = int(seg[e]), int(counts[e])
        assert torch.equal(d1[s:s + c], d[s:s + c])


def test_contiguous_and_masked_layouts_agree_bitwise(dev):
    counts = np.array([5, 64, 0, 33])
    E, N, K, max_m = 4, 256, 1024, 64
    (aq, asf, bq, sfb), _ = _operands(E * max_m, E, N, K, 91, dev)
    seg = np.arange(E + 1) * max_m
    dm = ops.grouped_gemm_masked(aq, asf, bq, sfb, torch.as_tensor(counts, dtype=torch.int32, device=dev), max_m)
    dc = ops.grouped_gemm_contig(aq, asf, bq, sfb, torch.as_tensor(seg, dtype=torch.int32, device=dev),
                                 torch.as_tensor(counts, dtype=torch.int32, device=dev))
    for e in range(E):
        s, c = int(seg[e]), int(counts[e])
        assert torch.equal(dm[s:s + c], dc[s:s + c])


def _workload_gemm_check(dev, name, n_sample=None, second=False):
    w = W.WORKLOADS[name]
    ids, _ = W.routing(w)
    K, N = (w.K2, w.N2) if second else (w.K, w.N)
    ref_r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align, max_m=w.max_m)
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    bufs = ops.route(ids.to(dev), w.E, w.layout, a_or_m)
    m_rows = bufs.m_cap
    x = W.activations(W.with_tokens(w, m_rows), device=dev, K=K, tag=1 if second else 0)
    aq, asf = ops.quantise_act(x)
    wt = W.weights(w, device=dev, N=N, K=K, tag=1 if second else 0)
    bq, sf128 = ops.quantise_weight(wt)
    sfb = ops.prepare_weight_sf(sf128, K)
    if w.layout == W.MASKED:
        d = ops.grouped_gemm_masked(aq, asf, bq, sfb, bufs.counts, w.max_m)
    else:
        d = ops.grouped_gemm_contig(aq, asf, bq, sfb, bufs.seg_start, bufs.counts)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    counts, seg = ref_r["counts"], ref_r["seg_start"]
    assert np.array_equal(i32(bufs.counts), counts)
    active = [e for e in range(w.E) if counts[e] > 0]
    if n_sample is not None:
        by_size = sorted(active, key=lambda e: counts[e])
        rng = np.random.default_rng(0)
        pick = {by_size[0], by_size[-1]} | set(rng.choice(active, n_sample, replace=False).tolist())
        active = sorted(pick)
    dg = bits16(d)
    for e in active:
        s, c = int(seg[e]), int(counts[e])
        a_ref, asf_ref = oracle.quantise.quantise_act(bits16(x[s:s + c]))
        b_ref, bsf_ref = oracle.quantise.quantise_weight(bits16(wt[e:e + 1]))
        assert np.array_equal(u8(aq[s:s + c]), a_ref)
        ref = oracle.gemm.expert_gemm(a_ref, asf_ref, b_ref[0], bsf_ref[0])
        check_expert_block(dg[s:s + c], ref, f"{name} expert {e} ({c} rows)")
    return d


def test_tiny_full(dev):
    _workload_gemm_check(dev, "tiny")
    _workload_gemm_check(dev, "tiny_a128")


def test_decode_full_size_sampled(dev):
    _workload_gemm_check(dev, "decode", n_sample=14)


def test_prefill_full_size_sampled(dev):
    _workload_gemm_check(dev, "prefill", n_sample=6)
    _workload_gemm_check(dev, "prefill", n_sample=6, second=True)


def test_large_full_size_sampled(dev):
    _workload_gemm_check(dev, "large", n_sample=6)
    _workload_gemm_check(dev, "large", n_sample=6, second=True)


def test_bitwise_determinism_20_runs(dev):
    counts = np.array([3, 200, 17, 0, 64, 9, 300, 1])
    E, N, K = len(counts), 512, 2048
    seg = np.concatenate([[0], np.cumsum(counts)])
    (aq, asf, bq, sfb), _ = _operands(int(seg[-1]), E, N, K, 5, dev)
    segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    first = ops.grouped_gemm_contig(aq, asf, bq, sfb, segt, ct)
    for _ in range(19):
        again = ops.grouped_gemm_contig(aq, asf, bq, sfb, segt, ct)
        assert torch.equal(again.view(torch.int16)[:int(seg[-1])], first.view(torch.int16)[:int(seg[-1])])
