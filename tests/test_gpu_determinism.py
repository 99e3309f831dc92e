"""Bitwise determinism over 20 repeated steps for every operand format (DeepGEMM article,
"精度与吞吐的平衡点": the same input run 20 times must give bit-identical output): routing is stable,
the GEMM tiles are statically scheduled, and no kernel on the path accumulates with atomics."""

import pytest
import torch

import workloads as W
from block_scaled_fp8_route_gb300 import MoEPath, ops
from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu

SMALL_DECODE = W.Workload("decode_small", T=128, kr=8, E=128, K=1024, N=256, layout=W.MASKED, max_m=64, seed=1001)
SMALL_PREFILL = W.Workload("prefill_small", T=512, kr=8, E=32, K=1024, N=512, layout=W.CONTIGUOUS, align=128,
                           routing="zipf", seed=1002)
# above the single-launch limit: multi-chunk routing (count -> assign) and, for FP8, the fused
# route + quantise-scatter path
MID_PREFILL = W.Workload("prefill_mid", T=4096, kr=8, E=64, K=1024, N=512, layout=W.CONTIGUOUS, align=128,
                         routing="zipf", seed=1003)


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4", "bf16", "fp8_f32sf"])
@pytest.mark.parametrize("w", [SMALL_DECODE, SMALL_PREFILL, MID_PREFILL], ids=["decode", "prefill", "prefill_mid"])
def test_twenty_runs_bit_identical(dev, fmt, w):
    x, wt = W.activations(w).to(dev), W.weights(w)
    ids, p = W.routing(w)
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=a_or_m, device=dev,
                   expected_m=w.T * w.kr // w.E, fmt=fmt)
    ids, p = ids.to(dev), p.to(dev)
    first = path.step(x, ids, p).clone()
    for _ in range(19):
        assert torch.equal(path.step(x, ids, p).view(torch.int16), first.view(torch.int16))
    assert ops.device_error() == 0
