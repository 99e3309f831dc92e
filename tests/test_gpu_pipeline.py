"""GPU parity of the combine kernel and of the whole path (quantise -> route ->
grouped GEMM -> combine) against the oracle."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from block_scaled_fp8_route_gb300 import MoEPath, ops
from tests.gpu_util import (bits16, check_combine_of_own_y, check_combined, check_expert_block, expert_row_rms, i32,
                            require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


@pytest.mark.parametrize("T,kr,rows,N", [(1, 1, 4, 8), (77, 8, 700, 3072), (513, 2, 1100, 264)])
def test_combine_within_one_ulp_of_float64(dev, T, kr, rows, N):
    g = torch.Generator().manual_seed(T)
    y = torch.randn(rows, N, generator=g).to(torch.bfloat16)
    idx = torch.randint(-1, rows, (T, kr), generator=g, dtype=torch.int32)
    p = torch.rand(T, kr, generator=g)
    z = ops.combine(y.to(dev), idx.to(dev), p.to(dev))
    torch.cuda.synchronize()
    ref = oracle.combine.combine(bits16(y), idx.numpy(), p.numpy())
    zg = bits16(z).astype(np.int64)
    # same sign-magnitude ordering: at most one bf16 step apart
    def ordered(b):
        b = b.astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    assert np.max(np.abs(ordered(zg) - ordered(ref))) <= 1


def _oracle_path(x, wt, ids, p, w, a_or_m):
    aq, asf = oracle.quantise.quantise_act(bits16(x))
    bq, bsf = oracle.quantise.quantise_weight(bits16(wt))
    r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align if w.layout == W.CONTIGUOUS else 1,
                           max_m=a_or_m if w.layout == W.MASKED else 0)
    a_rows = oracle.route.scatter_rows(aq, r["token_of_row"])
    a_sf = oracle.route.scatter_rows(asf, r["token_of_row"], pad_value=127)
    y, _ = oracle.gemm.grouped_gemm(a_rows, a_sf, bq, bsf, r["seg_start"], r["counts"])
    z = oracle.combine.combine(y, r["output_index"], p.numpy())
    return r, y, z


@pytest.mark.parametrize("name", ["tiny", "tiny_a128", "decode"])
def test_end_to_end(dev, name):
    w = W.WORKLOADS[name]
    x, wt = W.activations(w), W.weights(w)
    ids, p = W.routing(w)
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=a_or_m, device=dev,
                   expected_m=w.T * w.kr // w.E)
    z = path.step(x.to(dev), ids.to(dev), p.to(dev))
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    r, y_ref, z_ref = _oracle_path(x, wt, ids, p, w, a_or_m)
    assert np.array_equal(i32(path.bufs.output_index), r["output_index"])
    yg = bits16(path.y)
    for e in range(w.E):
        s, c = int(r["seg_start"][e]), int(r["counts"][e])
        if c:
            check_expert_block(yg[s:s + c], y_ref[s:s + c], f"{name} expert {e}")
    rms = expert_row_rms(y_ref, r["seg_start"], r["counts"])
    check_combined(bits16(z), z_ref, y_ref, r["output_index"], p.numpy(), rms, f"{name} combined output")
    # combine of the GPU's own y against the float64 combine of that y
    check_combine_of_own_y(bits16(z), yg, r["output_index"], p.numpy(), f"{name} combine")


def test_end_to_end_deterministic(dev):
    w = W.WORKLOADS["decode"]
    x, wt = W.activations(w), W.weights(w)
    ids, p = W.routing(w)
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=w.max_m, device=dev)
    xs, idss, ps = x.to(dev), ids.to(dev), p.to(dev)
    first = path.step(xs, idss, ps).clone()
    for _ in range(19):
        assert torch.equal(path.step(xs, idss, ps).view(torch.int16), first.view(torch.int16))


@pytest.mark.parametrize("name", ["decode", "tiny_a128"])
def test_graph_replay_matches_eager_step(dev, name):
    w = W.WORKLOADS[name]
    x, wt = W.activations(w).to(dev), W.weights(w)
    ids, p = W.routing(w)
    ids, p = ids.to(dev), p.to(dev)
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=a_or_m, device=dev)
    eager = path.step(x, ids, p).clone()
    path.capture(x, ids, p)
    # the graph holds its input tensors, so a caller dropping them cannot free memory it reads
    assert path._graph_inputs[0] is x and path._graph_inputs[1] is ids and path._graph_inputs[2] is p
    for _ in range(3):
        assert torch.equal(path.replay().view(torch.int16), eager.view(torch.int16))
    # new inputs written into the captured buffers are picked up by the replay
    x2 = W.activations(W.Workload(**{**w.__dict__, "seed": w.seed + 1})).to(dev)
    x.copy_(x2)
    expect = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=a_or_m,
                     device=dev).step(x2, ids, p)
    assert torch.equal(path.replay().view(torch.int16), expect.view(torch.int16))
    assert ops.device_error() == 0


def test_host_streamed_path_matches_eager_steps(dev):
    from block_scaled_fp8_route_gb300 import HostStreamedPath
    w = W.WORKLOADS["decode"]
    wt = W.weights(w)
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=w.max_m, device=dev)
    batches, expect = [], []
    for b in range(5):
        wb = W.Workload(**{**w.__dict__, "seed": w.seed + 7 * (b + 1)})
        x = W.activations(wb)
        ids, p = W.routing(wb)
        batches.append((x.pin_memory(), ids.pin_memory(), p.pin_memory()))
        expect.append(path.step(x.to(dev), ids.to(dev), p.to(dev)).cpu())
    streamed = HostStreamedPath(path, w.T, w.K, w.kr, device=dev)
    outs = [torch.empty(expect[0].shape, dtype=torch.bfloat16).pin_memory() for _ in batches]
    streamed.run(batches, outs)
    torch.cuda.synchronize()
    for got, exp in zip(outs, expect):
        assert torch.equal(got.view(torch.int16), exp.view(torch.int16))
    assert ops.device_error() == 0
