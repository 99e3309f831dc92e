"""Single-launch dispatch (quantise + route + scatter) for small batches: every
output is bit-identical to quantise_act followed by route with the scatter,
and to the oracle's routing."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from block_scaled_fp8_route_gb300 import _lib, ops
from tests.gpu_util import bits16, i32, require_gpu, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _compare(dev, x, ids, E, layout, a_or_m, check_oracle=True):
    x, ids = x.to(dev), torch.as_tensor(ids, dtype=torch.int32).to(dev)
    q, sf = ops.quantise_act(x)
    ref = ops.route(ids, E, layout, a_or_m, q=q, sf=sf)
    err_ref = ops.device_error()
    got = ops.dispatch(x, ids, E, layout, a_or_m)
    torch.cuda.synchronize()
    err_got = ops.device_error()
    assert err_got == err_ref
    for key in ("counts", "seg_start", "output_index"):
        assert torch.equal(getattr(got, key), getattr(ref, key)), key
    used = int(ref.seg_start[-1])
    for key in ("token_of_row", "m_indices"):
        assert torch.equal(getattr(got, key)[:used], getattr(ref, key)[:used]), key
    routed = ref.token_of_row[:used] >= 0
    assert torch.equal(got.a_packed[:used][routed], ref.a_packed[:used][routed])
    assert torch.equal(got.sfa_packed[:, :used][:, routed], ref.sfa_packed[:, :used][:, routed])
    if check_oracle:     # and the routing agrees with the oracle
        r = oracle.route.route(ids.cpu().numpy(), E, layout, align=a_or_m, max_m=a_or_m)
        assert np.array_equal(i32(got.output_index), r["output_index"])
    return got, err_got


@pytest.mark.parametrize("name", ["tiny", "tiny_a128", "decode"])
def test_dispatch_matches_three_step_path(dev, name):
    w = W.WORKLOADS[name]
    ids, _ = W.routing(w)
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    got, err = _compare(dev, W.activations(w), ids, w.E, w.layout, a_or_m)
    assert err == 0
    # the packed rows are the oracle's quantisation of the routed tokens
    aq, _ = oracle.quantise.quantise_act(bits16(W.activations(w)))
    r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align, max_m=w.max_m)
    tok = r["token_of_row"]
    rows = np.nonzero(tok >= 0)[0]
    assert np.array_equal(u8(got.a_packed)[rows], aq[tok[rows]])


@pytest.mark.parametrize("seed", range(5))
def test_dispatch_random_small_batches(dev, seed):
    rng = np.random.default_rng(100 + seed)
    T, kr = int(rng.integers(1, 1500)), int(rng.integers(1, 9))
    T = min(T, 16384 // kr)
    E = int(rng.integers(1, 257))
    K = int(rng.choice([128, 640, 1536]))
    ids = rng.integers(-1, E, (T, kr)).astype(np.int32)
    x = (torch.randn(T, K, generator=torch.Generator().manual_seed(seed)) * 3).to(torch.bfloat16)
    for layout, a in ((ops.CONTIGUOUS, 1), (ops.CONTIGUOUS, 128), (ops.MASKED, 16), (ops.MASKED, 256)):
        _compare(dev, x, ids, E, layout, a)


def test_dispatch_reports_overflow_bad_ids_and_rejects_large_batches(dev):
    x = torch.randn(4, 256).to(torch.bfloat16)
    ids = np.array([[0, 1], [0, 1], [0, 2], [1, 0]], dtype=np.int32)
    _, err = _compare(dev, x, ids, 3, ops.MASKED, 2)          # expert 0 and 1 overflow two slots
    assert err == ops.DEVERR_MASKED_OVERFLOW
    ids_bad = np.array([[0, 5], [1, 2], [2, -1], [7, 0]], dtype=np.int32)
    _, err = _compare(dev, x, ids_bad, 3, ops.CONTIGUOUS, 1, check_oracle=False)
    assert err == ops.DEVERR_EXPERT_ID
    big = torch.zeros((4096, 128), dtype=torch.bfloat16, device=dev)
    with pytest.raises(_lib.BsfError):
        ops.dispatch(big, torch.zeros((4096, 8), dtype=torch.int32, device=dev), 128, ops.CONTIGUOUS, 1)


def test_dependent_gemm_sees_the_dispatch_of_the_same_step(dev):
    """The small-batch GEMM starts as a programmatic dependent of the dispatch before it; back-to-back
    steps on alternating batches must give exactly what the same calls give with a full
    synchronisation between every launch."""
    E, K, N, T, kr, max_m = 16, 512, 256, 64, 4, 64
    g = torch.Generator().manual_seed(7)
    batches = []
    for _ in range(2):
        x = torch.randn(T, K, generator=g).to(torch.bfloat16).to(dev)
        ids = torch.stack([torch.randperm(E, generator=g)[:kr] for _ in range(T)]).to(torch.int32).to(dev)
        batches.append((x, ids))
    wq, sf128 = ops.quantise_weight((torch.randn(E, N, K, generator=g) * 0.02).to(torch.bfloat16).to(dev))
    sfb = ops.prepare_weight_sf(sf128, K)

    def step(x, ids, bufs, d, sync):
        ops.dispatch(x, ids, E, ops.MASKED, max_m, bufs=bufs)
        if sync:
            torch.cuda.synchronize()
        ops.grouped_gemm_masked(bufs.a_packed, bufs.sfa_packed, wq, sfb, bufs.counts, max_m, d=d, expected_m=16)
        if sync:
            torch.cuda.synchronize()

    bufs = ops.RouteBuffers(T, kr, E, ops.MASKED, max_m, K=K, device=dev)
    d = torch.empty((E * max_m, N), dtype=torch.bfloat16, device=dev)
    refs = []
    for x, ids in batches:
        step(x, ids, bufs, d, sync=True)
        refs.append((d.clone(), bufs.counts.clone()))
    outs = []
    for i in range(20):
        x, ids = batches[i % 2]
        step(x, ids, bufs, d, sync=False)
        outs.append(d.clone())                     # stream-ordered copy after the GEMM
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    for i, out in enumerate(outs):
        ref, counts = refs[i % 2]
        for e in range(E):
            rows = slice(e * max_m, e * max_m + int(counts[e]))
            assert torch.equal(out[rows].view(torch.int16), ref[rows].view(torch.int16)), (i, e)
