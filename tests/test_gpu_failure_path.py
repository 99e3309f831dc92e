"""Failure detection without a GPU fault: every spin in the GEMM kernel is
bounded.  With BSF_DEBUG_WITHHOLD_LOADS the load producer never fills a stage,
so each consumer's wait runs out after its limit (about 2 s); the kernel must
report BSF_DEVERR_TIMEOUT through the device error word, release its tensor
memory and return, leaving the CUDA context usable for the next call."""

import time

import numpy as np
import pytest
import torch

from block_scaled_fp8_route_gb300 import ops
from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu

WITHHOLD_LOADS = 0x100
TIMEOUT_BIT = 0x4


def _operands(dev, E=3, N=256, K=512, rows=96):
    g = torch.Generator().manual_seed(1)
    x = torch.randn(rows, K, generator=g).to(torch.bfloat16).to(dev)
    w = (torch.randn(E, N, K, generator=g) * 0.02).to(torch.bfloat16).to(dev)
    aq, asf = ops.quantise_act(x)
    bq, sf128 = ops.quantise_weight(w)
    return aq, asf, bq, ops.prepare_weight_sf(sf128, K)


@pytest.mark.parametrize("layout", ["contiguous", "masked"])
def test_withheld_loads_time_out_and_context_survives(layout):
    dev = require_gpu()
    aq, asf, bq, sfb = _operands(dev)
    counts = torch.tensor([32, 0, 64], dtype=torch.int32, device=dev)
    seg = torch.tensor([0, 32, 32, 96], dtype=torch.int32, device=dev)

    if layout == "masked":                            # 3 slots of 64 rows
        aq, asf, bq, sfb = _operands(dev, rows=3 * 64)
    rows = aq.shape[0]

    def run(flags, d):
        if layout == "masked":
            return ops.grouped_gemm_masked(aq, asf, bq, sfb, counts, 64, d=d, flags=flags)
        return ops.grouped_gemm_contig(aq, asf, bq, sfb, seg, counts, d=d, flags=flags)
    ref = run(0, torch.zeros((rows, 256), dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    assert ops.device_error() == 0

    sentinel = torch.full((rows, 256), 7.0, dtype=torch.bfloat16, device=dev)
    t0 = time.time()
    run(WITHHOLD_LOADS, sentinel)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    err = ops.device_error()
    assert err & TIMEOUT_BIT, f"expected the timeout bit, got {err:#x}"
    assert elapsed < 30, elapsed                       # bounded: the kernel gave up and returned
    assert torch.all(sentinel == 7.0)                  # nothing was written

    # the context is still usable and the next call is correct
    again = run(0, torch.zeros((rows, 256), dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
