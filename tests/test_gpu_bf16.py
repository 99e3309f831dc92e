"""GPU parity of the BF16 grouped GEMM (kind::f16) and the BF16 path against oracle/bf16.py.

Tolerance: the DeepGEMM article's BF16 threshold (calc_diff <= 1e-5, "精度与吞吐的平衡点") per
expert, plus the per-element bound of the FP8 checks (the FP32 accumulation moves a bf16 result by
at most about one step).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from block_scaled_fp8_route_gb300 import MoEPath, ops
from tests.gpu_util import bits16, check_combined, check_expert_block, expert_row_rms, i32, require_gpu

pytestmark = pytest.mark.gpu

CALC_DIFF_BF16 = 1e-5


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _operands(rows, E, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(rows, K, generator=g) * torch.exp2(torch.randint(-4, 5, (rows, 1), generator=g).float()))
    w = torch.randn(E, N, K, generator=g) * 0.02
    return x.to(torch.bfloat16), w.to(torch.bfloat16)


def _check(d, x, w, seg, counts, what):
    ref, _ = oracle.bf16.grouped_gemm(bits16(x), bits16(w), seg, counts)
    dg = bits16(d)
    for e in range(len(counts)):
        c, s = int(counts[e]), int(seg[e])
        if not c:
            continue
        check_expert_block(dg[s:s + c], ref[s:s + c], f"{what} expert {e} ({c} rows)")
        diff = oracle.checks.calc_diff(oracle.formats.bf16_bits_to_f64(dg[s:s + c]),
                                       oracle.formats.bf16_bits_to_f64(ref[s:s + c]))
        assert diff <= CALC_DIFF_BF16, f"{what} expert {e}: calc_diff {diff:.2e}"


@pytest.mark.parametrize("max_m,expected_m", [(64, 0), (320, 0), (320, 16)])
def test_masked_ragged(dev, max_m, expected_m):
    masked = np.minimum(np.array([0, 1, 16, 63, 64, max_m // 2, max_m, 7]), max_m)
    E, N, K = len(masked), 384, 576
    x, w = _operands(E * max_m, E, N, K, max_m + expected_m)
    d = torch.full((E * max_m, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_bf16_masked(x.to(dev), w.to(dev), torch.as_tensor(masked, dtype=torch.int32, device=dev),
                                 max_m, d=d, expected_m=expected_m)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check(d, x, w, np.arange(E + 1) * max_m, masked, f"bf16 masked max_m={max_m}")


@pytest.mark.parametrize("align", [1, 128])
def test_contig_ragged(dev, align):
    counts = np.array([1, 15, 16, 17, 31, 33, 0, 255, 256, 257, 600, 2])
    E, N, K = len(counts), 256, 1024
    seg = np.concatenate([[0], np.cumsum((counts + align - 1) // align * align)])
    rows = int(seg[-1])
    x, w = _operands(rows, E, N, K, 40 + align)
    d = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_bf16_contig(x.to(dev), w.to(dev), torch.as_tensor(seg, dtype=torch.int32, device=dev),
                                 torch.as_tensor(counts, dtype=torch.int32, device=dev), d=d)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check(d, x, w, seg, counts, f"bf16 contig align={align}")
    dv = d.float().cpu().numpy()
    for e in range(E):
        assert np.isnan(dv[seg[e] + counts[e]:seg[e + 1]]).all()


def test_weights_in_pinned_host_memory(dev):
    counts = np.array([5, 0, 300, 40])
    E, N, K = len(counts), 256, 512
    seg = np.concatenate([[0], np.cumsum(counts)])
    x, w = _operands(int(seg[-1]), E, N, K, 50)
    wh = w.pin_memory()
    segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    d_host = ops.grouped_gemm_bf16_contig(x.to(dev), wh, segt, ct, flags=ops.B_HOST_MAPPED)
    d_dev = ops.grouped_gemm_bf16_contig(x.to(dev), w.to(dev), segt, ct)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check(d_host, x, w, seg, counts, "bf16 host weights")
    for e in range(E):
        s, c = int(seg[e]), int(counts[e])
        assert torch.equal(d_host[s:s + c].view(torch.int16), d_dev[s:s + c].view(torch.int16))


def test_route_bf16_scatters_rows(dev):
    w = W.WORKLOADS["tiny_a128"]
    ids, _ = W.routing(w)
    x = W.activations(w)
    bufs = ops.route(ids.to(dev), w.E, w.layout, w.align, q=x.to(dev), fmt="bf16")
    torch.cuda.synchronize()
    r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align)
    assert np.array_equal(i32(bufs.output_index), r["output_index"])
    tok = r["token_of_row"]
    rows = np.nonzero(tok >= 0)[0]
    assert np.array_equal(bits16(bufs.a_packed)[rows], bits16(x)[tok[rows]])


DECODE_SMALL = W.Workload("decode_small", T=128, kr=8, E=128, K=1024, N=256, layout=W.MASKED, max_m=64, seed=1001)


@pytest.mark.parametrize("name", ["tiny", "tiny_a128", "decode_small"])
def test_bf16_end_to_end(dev, name):
    w = DECODE_SMALL if name == "decode_small" else W.WORKLOADS[name]
    x, wt = W.activations(w), W.weights(w)
    ids, p = W.routing(w)
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=a_or_m, device=dev,
                   expected_m=w.T * w.kr // w.E, fmt="bf16")
    z = path.step(x.to(dev), ids.to(dev), p.to(dev))
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align if w.layout == W.CONTIGUOUS else 1,
                           max_m=a_or_m if w.layout == W.MASKED else 0)
    a_rows = oracle.route.scatter_rows(bits16(x), r["token_of_row"])
    y_ref, _ = oracle.bf16.grouped_gemm(a_rows, bits16(wt), r["seg_start"], r["counts"])
    z_ref = oracle.combine.combine(y_ref, r["output_index"], p.numpy())
    yg = bits16(path.y)
    for e in range(w.E):
        s, c = int(r["seg_start"][e]), int(r["counts"][e])
        if c:
            check_expert_block(yg[s:s + c], y_ref[s:s + c], f"bf16 {name} expert {e}")
    rms = expert_row_rms(y_ref, r["seg_start"], r["counts"])
    check_combined(bits16(z), z_ref, y_ref, r["output_index"], p.numpy(), rms, f"bf16 {name} combined")


def test_masked_many_experts(dev):
    """More than 256 experts: the small-slot tile with 1024-expert tables."""
    rng = np.random.default_rng(7)
    E, N, K, max_m = 260, 128, 128, 32
    masked = rng.integers(0, max_m + 1, E)
    x, w = _operands(E * max_m, E, N, K, 70)
    d = torch.full((E * max_m, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_bf16_masked(x.to(dev), w.to(dev), torch.as_tensor(masked, dtype=torch.int32, device=dev),
                                 max_m, d=d)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check(d, x, w, np.arange(E + 1) * max_m, masked, "bf16 masked E=260")


def test_route_bf16_above_the_single_launch_limit(dev):
    rng = np.random.default_rng(8)
    T, kr, E, K = 2500, 8, 64, 256
    ids = np.stack([rng.permutation(E)[:kr] for _ in range(T)]).astype(np.int32)
    x, _ = _operands(T, 1, 128, K, 71)
    bufs = ops.route(torch.from_numpy(ids).to(dev), E, ops.CONTIGUOUS, 128, q=x.to(dev), fmt="bf16")
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    r = oracle.route.route(ids, E, ops.CONTIGUOUS, align=128)
    assert np.array_equal(i32(bufs.output_index), r["output_index"])
    tok = r["token_of_row"]
    rows = np.nonzero(tok >= 0)[0]
    assert np.array_equal(bits16(bufs.a_packed)[rows], bits16(x)[tok[rows]])
