"""GPU parity: quantisers, weight-SF transform and routing are bit-exact with the oracle.

Quantised codes are decided in the same precision on both sides: the scale
exponent is an exact integer function of amax, the scaled value x * 2**-e is
exact, and E4M3 rounding is nearest-even on the exact value.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from block_scaled_fp8_route_gb300 import ops
from tests.gpu_util import bits16, i32, require_gpu, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _x(T, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, K, generator=g) * torch.exp2(torch.randint(-20, 20, (T, 1), generator=g).float())
    if T > 3:
        x[1] = 0.0                                  # all-zero row: scale byte 127
        x[2, :128] *= 1e-30                         # tiny block
        x[3, 5] = 3.0e38                            # huge single value
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("T,K", [(1, 128), (37, 640), (128, 4096), (300, 1536), (8, 7168)])
def test_quantise_act_bit_exact(dev, T, K):
    x = _x(T, K, T * 1000 + K)
    q, sf = ops.quantise_act(x.to(dev))
    torch.cuda.synchronize()
    q_ref, sf_bytes = oracle.quantise.quantise_act(bits16(x))
    assert np.array_equal(u8(q), q_ref)
    sf_ref = oracle.quantise.pack_sf(sf_bytes)
    assert np.array_equal(sf.cpu().numpy()[:, :T], sf_ref[:, :T])


def test_quantise_weight_and_prepare_bit_exact(dev):
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(3, 256, 640, generator=g) * 0.02)
    w[1, 130:140, 300:310] *= 1e4
    w = w.to(torch.bfloat16)
    q, sf128 = ops.quantise_weight(w.to(dev))
    sfb = ops.prepare_weight_sf(sf128, 640)
    torch.cuda.synchronize()
    q_ref, sf_ref = oracle.quantise.quantise_weight(bits16(w))
    assert np.array_equal(u8(q), q_ref)
    assert np.array_equal(sf128.cpu().numpy().view(np.uint32), sf_ref.view(np.uint32))
    assert np.array_equal(sfb.cpu().numpy(), oracle.quantise.prepare_weight_sf(sf_ref))
    assert ops.device_error() == 0


def test_prepare_weight_sf_flags_bad_scale(dev):
    sf = torch.ones(1, 1, 4)
    sf[0, 0, 2] = 3.0
    ops.prepare_weight_sf(sf.to(dev), 512)
    assert ops.device_error() & 0x8


def _route_gpu(dev, ids, E, layout, a_or_m, q=None, sf=None):
    bufs = ops.route(torch.as_tensor(ids, dtype=torch.int32).to(dev), E, layout, a_or_m,
                     q=q, sf=sf)
    torch.cuda.synchronize()
    return bufs


def _check_route(bufs, ref, layout):
    E = len(ref["counts"])
    assert np.array_equal(i32(bufs.counts), ref["counts"])
    assert np.array_equal(i32(bufs.seg_start), ref["seg_start"])
    assert np.array_equal(i32(bufs.output_index), ref["output_index"])
    used = ref["rows_used"]
    assert np.array_equal(i32(bufs.token_of_row)[:used], ref["token_of_row"])
    assert np.array_equal(i32(bufs.m_indices)[:used], ref["m_indices"])
    assert E == len(ref["seg_start"]) - 1


def test_route_worked_example(dev, golden_dir):
    with open(os.path.join(golden_dir, "routing_example_t5_kr2_e4.json")) as f:
        ex = json.load(f)
    for align in (1, 128):
        bufs = _route_gpu(dev, ex["topk_ids"], ex["E"], ops.CONTIGUOUS, align)
        key = "unaligned" if align == 1 else "aligned_128"
        assert i32(bufs.output_index).tolist() == ex[key]["output_index"]
        assert int(bufs.seg_start[-1]) == ex[key]["M_packed"]
        ref = oracle.route.route(ex["topk_ids"], ex["E"], oracle.route.CONTIGUOUS, align=align)
        _check_route(bufs, ref, ops.CONTIGUOUS)


@pytest.mark.parametrize("seed", range(6))
def test_route_random_with_duplicates_and_drops(dev, seed):
    rng = np.random.default_rng(seed)
    T, kr, E = int(rng.integers(1, 3000)), int(rng.integers(1, 9)), int(rng.integers(1, 300))
    ids = rng.integers(-1, E, (T, kr)).astype(np.int32)
    for layout, a in ((ops.CONTIGUOUS, 1), (ops.CONTIGUOUS, 128), (ops.MASKED, 4096)):
        ref = oracle.route.route(ids, E, layout, align=a, max_m=a)
        bufs = _route_gpu(dev, ids, E, layout, a)
        _check_route(bufs, ref, layout)
    assert ops.device_error() == 0


# the multi-CTA route picks 512-, 1024- or 2048-assignment chunks by batch size (at most 64 chunks,
# else 2048 and a separate scan): one batch in each regime, each with a ragged last chunk
@pytest.mark.parametrize("T,kr,E", [(2049, 8, 64), (4000, 8, 300), (5000, 8, 128), (9000, 8, 1024),
                                    (20001, 8, 256)])
def test_route_every_chunk_size(dev, T, kr, E):
    rng = np.random.default_rng(T)
    ids = rng.integers(-1, E, (T, kr)).astype(np.int32)
    for layout, a in ((ops.CONTIGUOUS, 128), (ops.MASKED, 2 * T * kr // E + 64)):
        ref = oracle.route.route(ids, E, layout, align=a, max_m=a)
        bufs = _route_gpu(dev, ids, E, layout, a)
        _check_route(bufs, ref, layout)
    assert ops.device_error() == 0


def test_route_masked_overflow_and_bad_id(dev):
    ids = np.array([[0, 1], [0, 1], [0, 2], [1, 0]], dtype=np.int32)
    ref = oracle.route.route(ids, 3, oracle.route.MASKED, max_m=2)
    bufs = _route_gpu(dev, ids, 3, ops.MASKED, 2)
    _check_route(bufs, ref, ops.MASKED)
    assert ops.device_error() == 0x2
    _route_gpu(dev, np.array([[0, 3]], dtype=np.int32), 3, ops.CONTIGUOUS, 1)
    assert ops.device_error() & 0x1


@pytest.mark.parametrize("name", ["tiny", "tiny_a128", "decode", "prefill", "large"])
def test_route_and_scatter_full_size(dev, name):
    w = W.WORKLOADS[name]
    ids, _ = W.routing(w)
    K = 512 if name in ("prefill", "large") else w.K     # scatter checked on a narrower row
    x = W.activations(W.with_tokens(w, w.T), K=K)
    q, sf = ops.quantise_act(x.to(dev))
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    bufs = _route_gpu(dev, ids.numpy(), w.E, w.layout, a_or_m, q=q, sf=sf)
    ref = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align, max_m=w.max_m)
    _check_route(bufs, ref, w.layout)
    assert int(ref["M"].sum()) == w.T * w.kr
    aq, asf = oracle.quantise.quantise_act(bits16(x))
    used = ref["rows_used"]
    routed = ref["token_of_row"] >= 0            # padding rows are left unwritten (uninitialised, §4.6)
    rows = oracle.route.scatter_rows(aq, ref["token_of_row"])
    sfb = oracle.route.scatter_rows(asf, ref["token_of_row"], pad_value=127)
    assert np.array_equal(u8(bufs.a_packed)[:used][routed], rows[routed])
    sfw = bufs.sfa_packed.cpu().numpy()[:, :used]
    assert np.array_equal(oracle.quantise.unpack_sf(sfw, used, K // 128)[routed], sfb[routed])
    assert ops.device_error() == 0


def test_quantise_act_rows_writes_exactly_the_routed_rows():
    """bsf_quantise_act_rows on a packed operand: routed rows bit-identical to bsf_quantise_act,
    padding rows and rows past the last segment (data and scale words) left as they were."""
    dev = require_gpu()
    w = W.WORKLOADS["prefill"]
    ids, _ = W.routing(w)
    bufs = ops.route(ids.to(dev), w.E, w.layout, w.align)
    K = 1536
    x = W.activations(W.with_tokens(w, bufs.m_cap), device=dev, K=K, tag=1)
    q_all, sf_all = ops.quantise_act(x)
    q = torch.full_like(q_all, 0xA5)
    sf = torch.full_like(sf_all, -3)
    ops.quantise_act(x, q=q, sf=sf, rows=(bufs.token_of_row, bufs.seg_start[w.E:]))
    torch.cuda.synchronize()
    used = int(bufs.seg_start[-1])
    tok = bufs.token_of_row[:used]
    routed = torch.zeros(bufs.m_cap, dtype=torch.bool, device=dev)
    routed[:used] = tok >= 0
    assert int(routed.sum()) == w.T * w.kr
    assert torch.equal(q[routed], q_all[routed])
    assert torch.equal(sf[:, :bufs.m_cap][:, routed], sf_all[:, :bufs.m_cap][:, routed])
    assert bool((q[~routed] == 0xA5).all()) and bool((sf[:, :bufs.m_cap][:, ~routed] == -3).all())
    assert ops.device_error() == 0


@pytest.mark.parametrize("name", ["tiny", "tiny_a128", "decode", "prefill", "large"])
def test_route_quantise_matches_oracle(dev, name):
    """bsf_route_quantise (route, then every token quantised once into its k_r packed rows): routing
    arrays, packed rows and scale words against the oracle, as for quantise + route."""
    w = W.WORKLOADS[name]
    ids, _ = W.routing(w)
    K = 512 if name in ("prefill", "large") else w.K
    x = W.activations(W.with_tokens(w, w.T), K=K)
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    bufs = ops.route_quantise(x.to(dev), ids.to(dev), w.E, w.layout, a_or_m)
    torch.cuda.synchronize()
    ref = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align, max_m=w.max_m)
    _check_route(bufs, ref, w.layout)
    aq, asf = oracle.quantise.quantise_act(bits16(x))
    used = ref["rows_used"]
    routed = ref["token_of_row"] >= 0
    rows = oracle.route.scatter_rows(aq, ref["token_of_row"])
    sfb = oracle.route.scatter_rows(asf, ref["token_of_row"], pad_value=127)
    assert np.array_equal(u8(bufs.a_packed)[:used][routed], rows[routed])
    sfw = bufs.sfa_packed.cpu().numpy()[:, :used]
    assert np.array_equal(oracle.quantise.unpack_sf(sfw, used, K // 128)[routed], sfb[routed])
    assert ops.device_error() == 0


@pytest.mark.parametrize("seed", range(4))
def test_route_quantise_equals_quantise_then_route(dev, seed):
    """Drops (-1), repeated experts, masked overflow, ragged K: every output of the fused path is
    bit-identical to bsf_quantise_act + bsf_route with the scatter; padding rows stay untouched."""
    rng = np.random.default_rng(100 + seed)
    T, kr, E = int(rng.integers(1, 5000)), int(rng.integers(1, 9)), int(rng.integers(1, 300))
    K = 128 * int(rng.integers(1, 12))
    ids = torch.as_tensor(rng.integers(-1, E, (T, kr)).astype(np.int32)).to(dev)
    x = _x(T, K, seed).to(dev)
    for layout, a in ((ops.CONTIGUOUS, 1), (ops.CONTIGUOUS, 128), (ops.MASKED, max(1, (T * kr) // (2 * E)))):
        q, sf = ops.quantise_act(x)
        ref = ops.route(ids, E, layout, a, q=q, sf=sf)
        got = ops.RouteBuffers(T, kr, E, layout, a, K=K, device=dev)
        got.a_packed.fill_(0x5A)
        got.sfa_packed.fill_(-7)
        ops.route_quantise(x, ids, E, layout, a, bufs=got)
        torch.cuda.synchronize()
        assert ops.device_error() == ref_err(layout, ids, E, a)
        for name in ("counts", "seg_start", "output_index"):
            assert torch.equal(getattr(got, name), getattr(ref, name)), name
        used = int(ref.seg_start[-1])
        assert torch.equal(got.token_of_row[:used], ref.token_of_row[:used])
        assert torch.equal(got.m_indices[:used], ref.m_indices[:used])
        routed = torch.zeros(got.m_cap, dtype=torch.bool, device=dev)
        routed[:used] = ref.token_of_row[:used] >= 0
        assert torch.equal(got.a_packed[routed], ref.a_packed[routed])
        assert torch.equal(got.sfa_packed[:, :got.m_cap][:, routed], ref.sfa_packed[:, :got.m_cap][:, routed])
        assert bool((got.a_packed[~routed] == 0x5A).all())
        assert bool((got.sfa_packed[:, :got.m_cap][:, ~routed] == -7).all())


def ref_err(layout, ids, E, a):
    """Device error bits the routing of these ids raises (masked overflow only; ids are < E)."""
    if layout != ops.MASKED:
        return 0
    counts = torch.bincount(ids[ids >= 0].long().flatten(), minlength=E)
    return 0x2 if bool((counts > a).any()) else 0
