"""GPU parity of the NVFP4 path against the oracle (oracle/nvfp4.py).

Quantisers, tensor exponents and dispatch are bit-exact; the grouped GEMM is
within the FP8 GEMM's tolerance (the same FP32 tensor-core accumulation);
the FP4 GEMM equals the FP8 GEMM on the same values where every sum is exact
(DeepGEMM article, "精度与吞吐的平衡点": FP4 / FP8 equivalence).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from block_scaled_fp8_route_gb300 import _lib, ops
from tests.gpu_util import bits16, check_expert_block, i32, require_gpu, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _x(rows, K, seed, scale_rows=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g)
    if scale_rows:
        x = x * torch.exp2(torch.randint(-6, 7, (rows, 1), generator=g).float())
    return x.to(torch.bfloat16)


def test_tensor_exponent_matches_oracle(dev):
    x = _x(64, 512, 1)
    x[3] = 0
    x[5, 7] = 3000.0
    groups = 8
    got = ops.nvfp4_tensor_exponent(x.to(dev), groups=groups).cpu().numpy()
    xv = oracle.formats.bf16_bits_to_f64(bits16(x)).reshape(groups, -1)
    assert np.array_equal(got, oracle.nvfp4.global_exponent(np.abs(xv).max(axis=1)))
    z = torch.zeros(1024, dtype=torch.bfloat16, device=dev)
    assert int(ops.nvfp4_tensor_exponent(z)[0]) == 0


@pytest.mark.parametrize("a_exp", [0, -4, 6])
def test_quantise_act_bit_exact(dev, a_exp):
    T, K = 37, 320                                   # ragged rows, K not a multiple of 256
    x = _x(T, K, 2 + a_exp)
    x[0] = 0                                          # all-zero blocks
    x[1, :16] = torch.tensor([6, 3, -1.5, 0.25, 0.75, -4, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, 0, 0.5, -6.0])
    x[2, :16] = 1e-30                                 # scale underflows to 0
    x[4, 16:32] = 60000.0                             # scale saturates
    q, sf = ops.quantise_act_nvfp4(x.to(dev), a_exp)
    torch.cuda.synchronize()
    q_ref, sf_ref, _ = oracle.nvfp4.quantise_act(bits16(x), a_exp)
    assert np.array_equal(u8(q), q_ref)
    assert np.array_equal(sf.cpu().numpy()[:, :T], sf_ref[:, :T])


def test_quantise_weight_bit_exact(dev):
    E, N, K = 3, 256, 512
    g = torch.Generator().manual_seed(3)
    w = (torch.randn(E, N, K, generator=g) * 0.02 * torch.tensor([1.0, 30.0, 0.001]).view(E, 1, 1)).to(torch.bfloat16)
    q, sfb, b_exp = ops.quantise_weight_nvfp4(w.to(dev))
    torch.cuda.synchronize()
    wv = oracle.formats.bf16_bits_to_f64(bits16(w))
    j_ref = oracle.nvfp4.global_exponent(np.abs(wv).reshape(E, -1).max(axis=1))
    assert np.array_equal(b_exp.cpu().numpy(), j_ref)
    q_ref, sfb_ref, _ = oracle.nvfp4.quantise_weight(bits16(w), j_ref)
    assert np.array_equal(u8(q), q_ref)
    assert np.array_equal(sfb.cpu().numpy(), sfb_ref)


def _gemm_operands(rows, E, N, K, seed, dev, a_exp=0):
    x = _x(rows, K, seed)
    g = torch.Generator().manual_seed(seed + 1)
    w = (torch.randn(E, N, K, generator=g) * 0.02).to(torch.bfloat16)
    aq, asf = ops.quantise_act_nvfp4(x.to(dev), a_exp)
    bq, sfb, b_exp = ops.quantise_weight_nvfp4(w.to(dev))
    aq_r, _, asc_r = oracle.nvfp4.quantise_act(bits16(x), a_exp)
    wv = oracle.formats.bf16_bits_to_f64(bits16(w))
    j_r = oracle.nvfp4.global_exponent(np.abs(wv).reshape(E, -1).max(axis=1))
    bq_r, _, bsc_r = oracle.nvfp4.quantise_weight(bits16(w), j_r)
    return (aq, asf, bq, sfb, b_exp), (aq_r, asc_r, a_exp, bq_r, bsc_r, j_r)


def _check(d, ref_ops, seg, counts, what):
    aq_r, asc_r, aj, bq_r, bsc_r, j_r = ref_ops
    ref, _ = oracle.nvfp4.grouped_gemm(aq_r, asc_r, aj, bq_r, bsc_r, j_r, seg, counts)
    dg = bits16(d)
    for e in range(len(counts)):
        c, s = int(counts[e]), int(seg[e])
        if c:
            check_expert_block(dg[s:s + c], ref[s:s + c], f"{what} expert {e} ({c} rows)")


@pytest.mark.parametrize("max_m,expected_m", [(64, 0), (200, 0)])
def test_masked_gemm(dev, max_m, expected_m):
    masked = np.minimum(np.array([0, 1, 16, 63, 64, max_m // 2, max_m, 7]), max_m)
    E, N, K = len(masked), 256, 512
    ops_, ref_ops = _gemm_operands(E * max_m, E, N, K, 10 + max_m, dev, a_exp=-1)
    aq, asf, bq, sfb, b_exp = ops_
    d = torch.full((E * max_m, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_nvfp4_masked(aq, asf, -1, bq, sfb, b_exp, torch.as_tensor(masked, dtype=torch.int32,
                                  device=dev), max_m, d=d, expected_m=expected_m)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check(d, ref_ops, np.arange(E + 1) * max_m, masked, f"nvfp4 masked max_m={max_m}")


@pytest.mark.parametrize("align,N", [(1, 384), (128, 384), (1, 512)])
def test_contig_gemm_ragged(dev, align, N):
    """N = 384: 128-row weight tiles; N = 512: 256-row work items (two weight tiles per token chunk)."""
    counts = np.array([1, 15, 16, 17, 31, 33, 0, 129, 250, 3])
    E, K = len(counts), 768
    seg = np.concatenate([[0], np.cumsum((counts + align - 1) // align * align)])
    rows = int(seg[-1])
    ops_, ref_ops = _gemm_operands(rows, E, N, K, 20 + align + N, dev)
    aq, asf, bq, sfb, b_exp = ops_
    d = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm_nvfp4_contig(aq, asf, 0, bq, sfb, b_exp, torch.as_tensor(seg, dtype=torch.int32, device=dev),
                                  torch.as_tensor(counts, dtype=torch.int32, device=dev), d=d)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    _check(d, ref_ops, seg, counts, f"nvfp4 contig align={align}")
    dv = d.float().cpu().numpy()
    for e in range(E):
        assert np.isnan(dv[seg[e] + counts[e]:seg[e + 1]]).all()


def test_fp4_gemm_equals_fp8_gemm_on_the_same_values(dev):
    """Every FP4 scale 1 and every sum exact in FP32: the two block-scaled MMA kinds must agree bit for bit."""
    rng = np.random.default_rng(11)
    R, E, N, K = 96, 2, 256, 1024
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    xa = rng.choice(grid, (R, K)) * rng.choice([-1, 1], (R, K))
    xb = rng.choice(grid, (E, N, K)) * rng.choice([-1, 1], (E, N, K))
    xa[:, ::16] = 6.0
    xb[:, :, ::16] = 6.0
    xa_t = torch.from_numpy(xa).to(torch.bfloat16).to(dev)
    xb_t = torch.from_numpy(xb).to(torch.bfloat16).to(dev)
    zeros = torch.zeros(E, dtype=torch.int32, device=dev)
    aq4, asf4 = ops.quantise_act_nvfp4(xa_t, 0)
    bq4, sfb4, _ = ops.quantise_weight_nvfp4(xb_t, zeros)
    counts = torch.tensor([60, 36], dtype=torch.int32, device=dev)
    seg = torch.tensor([0, 60, 96], dtype=torch.int32, device=dev)
    d4 = ops.grouped_gemm_nvfp4_contig(aq4, asf4, 0, bq4, sfb4, zeros, seg, counts)
    # FP8 operands holding the same values (every block's amax is 6: scale 2**-6, codes 64 x value, exact)
    aq8, asf8 = ops.quantise_act(xa_t)
    bq8, sf128 = ops.quantise_weight(xb_t)
    assert torch.all(sf128 == 2.0 ** -6)
    d8 = ops.grouped_gemm_contig(aq8, asf8, bq8, ops.prepare_weight_sf(sf128, K), seg, counts)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    assert torch.equal(d4.view(torch.int16), d8.view(torch.int16))


def test_dispatch_nvfp4_matches_quantise_and_scatter(dev):
    for name in ("tiny", "decode"):
        w = W.WORKLOADS[name]
        ids, _ = W.routing(w)
        x = W.activations(w)
        a_or_m = w.max_m if w.layout == W.MASKED else w.align
        got = ops.dispatch_nvfp4(x.to(dev), ids.to(dev), w.E, w.layout, a_or_m, a_exp=1)
        torch.cuda.synchronize()
        assert ops.device_error() == 0
        q_ref, sf_ref, _ = oracle.nvfp4.quantise_act(bits16(x), 1)
        r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align, max_m=w.max_m)
        assert np.array_equal(i32(got.output_index), r["output_index"])
        tok = r["token_of_row"]
        rows = np.nonzero(tok >= 0)[0]
        assert np.array_equal(u8(got.a_packed)[rows], q_ref[tok[rows]])
        assert np.array_equal(got.sfa_packed.cpu().numpy()[:, rows], sf_ref[:, tok[rows]])


def test_nvfp4_argument_checks(dev):
    a = torch.zeros((64, 64), dtype=torch.uint8, device=dev)        # K = 128: not a multiple of 256
    sfa = torch.zeros((2, 64), dtype=torch.int32, device=dev)
    b = torch.zeros((1, 128, 64), dtype=torch.uint8, device=dev)
    sfb = torch.zeros((1, 2, 128), dtype=torch.int32, device=dev)
    m = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(_lib.BsfError):
        ops.grouped_gemm_nvfp4_masked(a, sfa, 0, b, sfb, None, m, 64)
    with pytest.raises(_lib.BsfError):
        ops.quantise_act_nvfp4(torch.zeros((4, 64), dtype=torch.bfloat16, device=dev), a_exp=101)


def _exp_of(wt):
    wv = oracle.formats.bf16_bits_to_f64(bits16(wt))
    return oracle.nvfp4.global_exponent(np.abs(wv).reshape(wv.shape[0], -1).max(axis=1))


def test_decode_full_size_sampled(dev):
    """The decode workload's grouped GEMM at full size (128 experts, K 4096, N 3072), 14 sampled experts."""
    w = W.WORKLOADS["decode"]
    ids, _ = W.routing(w)
    r = oracle.route.route(ids.numpy(), w.E, w.layout, max_m=w.max_m)
    bufs = ops.route(ids.to(dev), w.E, w.layout, w.max_m)
    x = W.activations(W.with_tokens(w, bufs.m_cap), device=dev)
    aq, asf = ops.quantise_act_nvfp4(x, 0)
    wt = W.weights(w, device=dev)
    bq, sfb, b_exp = ops.quantise_weight_nvfp4(wt)
    d = ops.grouped_gemm_nvfp4_masked(aq, asf, 0, bq, sfb, b_exp, bufs.counts, w.max_m, expected_m=8)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    counts = r["counts"]
    active = [e for e in range(w.E) if counts[e] > 0]
    by_size = sorted(active, key=lambda e: counts[e])
    pick = sorted({by_size[0], by_size[-1]} | set(np.random.default_rng(0).choice(active, 12, replace=False).tolist()))
    dg = bits16(d)
    for e in pick:
        s, c = e * w.max_m, int(counts[e])
        aq_r, _, asc_r = oracle.nvfp4.quantise_act(bits16(x[s:s + c]), 0)
        assert np.array_equal(u8(aq[s:s + c]), aq_r)
        j = _exp_of(wt[e:e + 1])
        assert int(b_exp[e]) == int(j[0])
        bq_r, _, bsc_r = oracle.nvfp4.quantise_weight(bits16(wt[e:e + 1]), j)
        ref, _ = oracle.nvfp4.grouped_gemm(aq_r, asc_r, 0, bq_r, bsc_r, j, np.array([0, c]), np.array([c]))
        check_expert_block(dg[s:s + c], ref[:c], f"nvfp4 decode expert {e} ({c} rows)")


DECODE_SMALL = W.Workload("decode_small", T=128, kr=8, E=128, K=1024, N=256, layout=W.MASKED, max_m=64, seed=1001)


@pytest.mark.parametrize("name,fused", [("tiny", True), ("tiny_a128", False), ("decode_small", True),
                                        ("decode_small", False)])
def test_nvfp4_end_to_end(dev, name, fused):
    from block_scaled_fp8_route_gb300 import MoEPath
    from tests.gpu_util import check_combined, expert_row_rms
    w = DECODE_SMALL if name == "decode_small" else W.WORKLOADS[name]
    x, wt = W.activations(w), W.weights(w)
    ids, p = W.routing(w)
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=a_or_m, device=dev,
                   expected_m=w.T * w.kr // w.E, fused_dispatch=fused, fmt="nvfp4", a_exp=-1)
    z = path.step(x.to(dev), ids.to(dev), p.to(dev))
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    # oracle: quantise, route, scatter, NVFP4 grouped GEMM, combine
    aq, _, asc = oracle.nvfp4.quantise_act(bits16(x), -1)
    j = _exp_of(wt)
    bq, _, bsc = oracle.nvfp4.quantise_weight(bits16(wt), j)
    r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align if w.layout == W.CONTIGUOUS else 1,
                           max_m=a_or_m if w.layout == W.MASKED else 0)
    a_rows = oracle.route.scatter_rows(aq, r["token_of_row"])
    a_sc = oracle.route.scatter_rows(asc, r["token_of_row"])
    y_ref, _ = oracle.nvfp4.grouped_gemm(a_rows, a_sc, -1, bq, bsc, j, r["seg_start"], r["counts"])
    z_ref = oracle.combine.combine(y_ref, r["output_index"], p.numpy())
    assert np.array_equal(i32(path.bufs.output_index), r["output_index"])
    yg = bits16(path.y)
    for e in range(w.E):
        s, c = int(r["seg_start"][e]), int(r["counts"][e])
        if c:
            check_expert_block(yg[s:s + c], y_ref[s:s + c], f"nvfp4 {name} expert {e}")
    rms = expert_row_rms(y_ref, r["seg_start"], r["counts"])
    check_combined(bits16(z), z_ref, y_ref, r["output_index"], p.numpy(), rms, f"nvfp4 {name} combined")


def test_weights_in_pinned_host_memory_match_device_weights(dev):
    counts = np.array([5, 0, 130, 40])
    E, N, K = len(counts), 256, 512
    seg = np.concatenate([[0], np.cumsum(counts)])
    ops_, _ = _gemm_operands(int(seg[-1]), E, N, K, 60, dev)
    aq, asf, bq, sfb, b_exp = ops_
    segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    d_dev = ops.grouped_gemm_nvfp4_contig(aq, asf, 0, bq, sfb, b_exp, segt, ct)
    d_host = ops.grouped_gemm_nvfp4_contig(aq, asf, 0, bq.cpu().pin_memory(), sfb.cpu().pin_memory(), b_exp, segt, ct,
                                           flags=ops.B_HOST_MAPPED)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    for e in range(E):
        s, c = int(seg[e]), int(counts[e])
        assert torch.equal(d_host[s:s + c].view(torch.int16), d_dev[s:s + c].view(torch.int16))


def test_route_nvfp4_above_the_single_launch_limit(dev):
    """20000 assignments: the multi-block route path scatters the NVFP4 rows and scale words."""
    rng = np.random.default_rng(12)
    T, kr, E, K = 2500, 8, 64, 512
    ids = np.stack([rng.permutation(E)[:kr] for _ in range(T)]).astype(np.int32)
    x = _x(T, K, 13)
    q, sf = ops.quantise_act_nvfp4(x.to(dev), 0)
    bufs = ops.route(torch.from_numpy(ids).to(dev), E, ops.CONTIGUOUS, 128, q=q, sf=sf, fmt="nvfp4")
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    r = oracle.route.route(ids, E, ops.CONTIGUOUS, align=128)
    assert np.array_equal(i32(bufs.output_index), r["output_index"])
    tok = r["token_of_row"]
    rows = np.nonzero(tok >= 0)[0]
    q_ref, sf_ref, _ = oracle.nvfp4.quantise_act(bits16(x), 0)
    assert np.array_equal(u8(bufs.a_packed)[rows], q_ref[tok[rows]])
    assert np.array_equal(bufs.sfa_packed.cpu().numpy()[:, rows], sf_ref[:, tok[rows]])


@pytest.mark.parametrize("seed", range(3))
def test_dispatch_nvfp4_random_small_batches(dev, seed):
    rng = np.random.default_rng(200 + seed)
    T, kr = int(rng.integers(1, 1200)), int(rng.integers(1, 9))
    E = int(rng.integers(1, 257))
    K = int(rng.choice([64, 576, 1024]))
    ids = rng.integers(-1, E, (T, kr)).astype(np.int32)
    x = _x(T, K, 300 + seed)
    for layout, a in ((ops.CONTIGUOUS, 1), (ops.MASKED, 32)):
        got = ops.dispatch_nvfp4(x.to(dev), torch.from_numpy(ids).to(dev), E, layout, a, a_exp=2)
        torch.cuda.synchronize()
        r = oracle.route.route(ids, E, layout, align=a, max_m=a)
        assert np.array_equal(i32(got.output_index), r["output_index"])
        tok = r["token_of_row"]
        rows = np.nonzero(tok >= 0)[0]
        q_ref, sf_ref, _ = oracle.nvfp4.quantise_act(bits16(x), 2)
        assert np.array_equal(u8(got.a_packed)[rows], q_ref[tok[rows]])
        assert np.array_equal(got.sfa_packed.cpu().numpy()[:, rows], sf_ref[:, tok[rows]])
        ops.device_error()          # masked overflow is expected for some batches; clear it
