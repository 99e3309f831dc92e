"""GPU parity of the FP8 path with float32 scale factors (disable_ue8m0_cast) against oracle/f32sf.py.

Quantisers are bit-exact (codes and float32 scales); the grouped GEMM (per-128-K partials promoted
in FP32 on the CUDA cores) is within the FP8 GEMM's tolerance.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from block_scaled_fp8_route_gb300 import MoEPath, ops
from tests.gpu_util import bits16, check_combined, check_expert_block, expert_row_rms, i32, require_gpu, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _x(rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g) * torch.exp2(torch.randint(-8, 9, (rows, 1), generator=g).float())
    return x.to(torch.bfloat16)


def _w(E, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(E, N, K, generator=g) * 0.02).to(torch.bfloat16)


def test_quantisers_bit_exact(dev):
    x = _x(37, 640, 1)
    x[0] = 0
    q, sf = ops.quantise_act_f32sf(x.to(dev))
    w = _w(2, 256, 384, 2)
    wq, wsf = ops.quantise_weight_f32sf(w.to(dev))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.f32sf.quantise_act(bits16(x))
    assert np.array_equal(u8(q), q_ref)
    assert np.array_equal(sf.cpu().numpy()[:, :37], s_ref.T)
    wq_ref, ws_ref = oracle.f32sf.quantise_weight(bits16(w))
    assert np.array_equal(u8(wq), wq_ref)
    assert np.array_equal(wsf.cpu().numpy(), ws_ref)


def _ref(x, w, seg, counts):
    aq, as_ = oracle.f32sf.quantise_act(bits16(x))
    bq, bs = oracle.f32sf.quantise_weight(bits16(w))
    return oracle.f32sf.grouped_gemm(aq, as_, bq, bs, seg, counts)[0]


def _check(d, ref, seg, counts, what):
    dg = bits16(d)
    for e in range(len(counts)):
        c, s = int(counts[e]), int(seg[e])
        if c:
            check_expert_block(dg[s:s + c], ref[s:s + c], f"{what} expert {e} ({c} rows)")


@pytest.mark.parametrize("max_m,expected_m", [(64, 0), (64, 8), (32, 0), (200, 0), (200, 8)])
def test_masked(dev, max_m, expected_m):
    masked = np.minimum(np.array([0, 1, 16, 63, 64, max_m // 2, max_m, 7]), max_m)
    E, N, K = len(masked), 256, 512
    x, w = _x(E * max_m, K, 10 + max_m), _w(E, N, K, 11 + max_m)
    aq, asf = ops.quantise_act_f32sf(x.to(dev))
    bq, bsf = ops.quantise_weight_f32sf(w.to(dev))
    d = torch.full((E * max_m, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_f32sf_masked(aq, asf, bq, bsf, torch.as_tensor(masked, dtype=torch.int32, device=dev), max_m,
                                  d=d, expected_m=expected_m)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    seg = np.arange(E + 1) * max_m
    _check(d, _ref(x, w, seg, masked), seg, masked, f"f32sf masked max_m={max_m} expected_m={expected_m}")


@pytest.mark.parametrize("align", [1, 128])
def test_contig_ragged(dev, align):
    counts = np.array([1, 15, 16, 17, 31, 33, 0, 129, 250, 3])
    E, N, K = len(counts), 384, 768
    seg = np.concatenate([[0], np.cumsum((counts + align - 1) // align * align)])
    rows = int(seg[-1])
    x, w = _x(rows, K, 20 + align), _w(E, N, K, 21 + align)
    aq, asf = ops.quantise_act_f32sf(x.to(dev))
    bq, bsf = ops.quantise_weight_f32sf(w.to(dev))
    d = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_f32sf_contig(aq, asf, bq, bsf, torch.as_tensor(seg, dtype=torch.int32, device=dev),
                                  torch.as_tensor(counts, dtype=torch.int32, device=dev), d=d)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check(d, _ref(x, w, seg, counts), seg, counts, f"f32sf contig align={align}")
    dv = d.float().cpu().numpy()
    for e in range(E):
        assert np.isnan(dv[seg[e] + counts[e]:seg[e + 1]]).all()


def test_power_of_two_scales_match_the_ue8m0_gemm(dev):
    """UE8M0-quantised operands passed with their scales as float32: both GEMMs compute the same sum."""
    counts = np.array([9, 64, 0, 33])
    E, N, K = len(counts), 256, 1024
    seg = np.concatenate([[0], np.cumsum(counts)])
    rows = int(seg[-1])
    x, w = _x(rows, K, 30), _w(E, N, K, 31)
    aq, asf = ops.quantise_act(x.to(dev))
    bq, sf128 = ops.quantise_weight(w.to(dev))
    segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    d8 = ops.grouped_gemm_contig(aq, asf, bq, ops.prepare_weight_sf(sf128, K), segt, ct)
    # UE8M0 bytes -> float32 scales, MN-major [K/128][ld]
    words = asf.cpu().numpy().view(np.uint32)[:, :rows]
    by = np.stack([(words >> (8 * j)) & 0xFF for j in range(4)], axis=1).reshape(-1, rows)[:K // 128]
    sfa32 = np.zeros((K // 128, ops.sf_ld(rows)), dtype=np.float32)
    sfa32[:, :rows] = np.ldexp(1.0, by.astype(np.int64) - 127)
    d32 = ops.grouped_gemm_f32sf_contig(aq, torch.from_numpy(sfa32).to(dev), bq, sf128, segt, ct)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    aq_r, asf_r = oracle.quantise.quantise_act(bits16(x))
    bq_r, bsf_r = oracle.quantise.quantise_weight(bits16(w))
    ref, _ = oracle.gemm.grouped_gemm(aq_r, asf_r, bq_r, bsf_r, seg, counts)
    _check(d32, ref, seg, counts, "f32sf with power-of-two scales")
    _check(d8, ref, seg, counts, "ue8m0")


DECODE_SMALL = W.Workload("decode_small", T=128, kr=8, E=128, K=1024, N=256, layout=W.MASKED, max_m=64, seed=1001)


@pytest.mark.parametrize("name", ["tiny", "tiny_a128", "decode_small"])
def test_f32sf_end_to_end(dev, name):
    w = DECODE_SMALL if name == "decode_small" else W.WORKLOADS[name]
    x, wt = W.activations(w), W.weights(w)
    ids, p = W.routing(w)
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=a_or_m, device=dev,
                   expected_m=w.T * w.kr // w.E, fmt="fp8_f32sf")
    z = path.step(x.to(dev), ids.to(dev), p.to(dev))
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    aq, as_ = oracle.f32sf.quantise_act(bits16(x))
    bq, bs = oracle.f32sf.quantise_weight(bits16(wt))
    r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align if w.layout == W.CONTIGUOUS else 1,
                           max_m=a_or_m if w.layout == W.MASKED else 0)
    a_rows = oracle.route.scatter_rows(aq, r["token_of_row"])
    a_s = oracle.route.scatter_rows(as_, r["token_of_row"], pad_value=1.0)
    y_ref, _ = oracle.f32sf.grouped_gemm(a_rows, a_s, bq, bs, r["seg_start"], r["counts"])
    z_ref = oracle.combine.combine(y_ref, r["output_index"], p.numpy())
    assert np.array_equal(i32(path.bufs.output_index), r["output_index"])
    yg = bits16(path.y)
    for e in range(w.E):
        s, c = int(r["seg_start"][e]), int(r["counts"][e])
        if c:
            check_expert_block(yg[s:s + c], y_ref[s:s + c], f"f32sf {name} expert {e}")
    rms = expert_row_rms(y_ref, r["seg_start"], r["counts"])
    check_combined(bits16(z), z_ref, y_ref, r["output_index"], p.numpy(), rms, f"f32sf {name} combined")


def test_weights_in_pinned_host_memory_match_device_weights(dev):
    counts = np.array([5, 0, 70, 40])
    E, N, K = len(counts), 256, 512
    seg = np.concatenate([[0], np.cumsum(counts)])
    x, w = _x(int(seg[-1]), K, 80), _w(E, N, K, 81)
    aq, asf = ops.quantise_act_f32sf(x.to(dev))
    bq, bsf = ops.quantise_weight_f32sf(w.to(dev))
    segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    d_dev = ops.grouped_gemm_f32sf_contig(aq, asf, bq, bsf, segt, ct)
    d_host = ops.grouped_gemm_f32sf_contig(aq, asf, bq.cpu().pin_memory(), bsf.cpu().pin_memory(), segt, ct,
                                           flags=ops.B_HOST_MAPPED)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    for e in range(E):
        s, c = int(seg[e]), int(counts[e])
        assert torch.equal(d_host[s:s + c].view(torch.int16), d_dev[s:s + c].view(torch.int16))


def test_route_f32sf_above_the_single_launch_limit(dev):
    rng = np.random.default_rng(9)
    T, kr, E, K = 2500, 8, 64, 384
    ids = np.stack([rng.permutation(E)[:kr] for _ in range(T)]).astype(np.int32)
    x = _x(T, K, 82)
    q, sf = ops.quantise_act_f32sf(x.to(dev))
    bufs = ops.route(torch.from_numpy(ids).to(dev), E, ops.CONTIGUOUS, 1, q=q, sf=sf, fmt="fp8_f32sf")
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    r = oracle.route.route(ids, E, ops.CONTIGUOUS, align=1)
    tok = r["token_of_row"]
    rows = np.nonzero(tok >= 0)[0]
    q_ref, s_ref = oracle.f32sf.quantise_act(bits16(x))
    assert np.array_equal(u8(bufs.a_packed)[rows], q_ref[tok[rows]])
    assert np.array_equal(bufs.sfa_packed.cpu().numpy()[:, rows], s_ref.T[:, tok[rows]])
