"""bsf_route_no_alloc: routing without a caller-provided workspace.

Some callers cannot call cudaMalloc where they route: serving runtimes that
reserve all device memory at start-up, plug-ins whose host framework owns the
allocator, code inside an allocator callback.  This entry point keeps its
scratch in a fixed device array of the library.  Its outputs must equal those
of bsf_route (with a caller-allocated workspace) bit for bit — routing is
integer work — on two calls in a row, the second with different inputs so that
the first call's leftover scratch contents are exercised.  Both workloads are
large enough (T * k_r > 16384 assignments) to take the multi-block count /
scan / assign path, the one that uses the scratch array.  Collected last on
purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from block_scaled_fp8_route_gb300 import _lib, ops
from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 256 * 1024


def _bufs(T, kr, E, layout, a_or_m, K, dev):
    m_cap = ops.route_capacity(T, kr, E, layout, a_or_m)
    i32 = dict(dtype=torch.int32, device=dev)
    return {
        "counts": torch.full((E,), -7, **i32), "seg_start": torch.full((E + 1,), -7, **i32),
        "output_index": torch.full((T, kr), -7, **i32), "token_of_row": torch.full((m_cap,), -7, **i32),
        "m_indices": torch.full((m_cap,), -7, **i32),
        "a_packed": torch.full((m_cap, K), 0xAB, dtype=torch.uint8, device=dev),
        "sfa_packed": torch.full((ops.sf_words(K), ops.sf_ld(m_cap)), -7, **i32),
        "m_cap": m_cap,
    }


def _args(ids, E, layout, a_or_m, q, sf, b):
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    T, kr = ids.shape
    return [p(ids), T, kr, E, layout, a_or_m, p(b["counts"]), p(b["seg_start"]), p(b["output_index"]),
            p(b["token_of_row"]), p(b["m_indices"]), b["m_cap"], p(q), p(sf), sf.shape[1], q.shape[1],
            p(b["a_packed"]), p(b["sfa_packed"]), b["sfa_packed"].shape[1]]


def _compare(b_ref, b_new):
    used = int(b_ref["seg_start"][-1])
    for key in ("counts", "seg_start", "output_index"):
        assert torch.equal(b_ref[key], b_new[key]), key
    for key in ("token_of_row", "m_indices"):
        assert torch.equal(b_ref[key][:used], b_new[key][:used]), key
    routed = b_ref["token_of_row"][:used] >= 0          # padding rows are not written by either call
    assert torch.equal(b_ref["a_packed"][:used][routed], b_new["a_packed"][:used][routed])
    assert torch.equal(b_ref["sfa_packed"][:, :used][:, routed], b_new["sfa_packed"][:, :used][:, routed])


@pytest.mark.parametrize("name", ["large", "prefill"])
def test_no_alloc_route_matches_workspace_route_twice(name):
    dev = require_gpu()
    lib = _lib.load()
    w = W.WORKLOADS[name]
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    K = 512
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        wl = W.Workload(**{**w.__dict__, "seed": w.seed + 17 * call})
        ids, _ = W.routing(wl, device=dev)
        x = W.activations(wl, device=dev, K=K)
        q, sf = ops.quantise_act(x)
        assert w.T * w.kr > 16384              # above the single-CTA limit: count / scan / assign kernels
        ws = torch.empty(lib.bsf_route_workspace_bytes(w.T, w.kr, w.E), dtype=torch.uint8, device=dev)
        assert ws.numel() <= STATIC_SCRATCH_BYTES
        b_ref = _bufs(w.T, w.kr, w.E, w.layout, a_or_m, K, dev)
        b_new = _bufs(w.T, w.kr, w.E, w.layout, a_or_m, K, dev)
        _lib.check(lib.bsf_route(*_args(ids, w.E, w.layout, a_or_m, q, sf, b_ref),
                                 ctypes.c_void_p(ws.data_ptr()), ws.numel(), stream), "bsf_route")
        _lib.check(lib.bsf_route_no_alloc(*_args(ids, w.E, w.layout, a_or_m, q, sf, b_new), stream),
                   "bsf_route_no_alloc")
        torch.cuda.synchronize()
        _compare(b_ref, b_new)
    assert ops.device_error() == 0


def test_no_alloc_route_rejects_oversize_problems():
    require_gpu()
    lib = _lib.load()
    T, kr, E = 65536, 8, 1024          # 256 chunks x 1024 experts x 4 B = 1 MiB > 256 KiB
    assert lib.bsf_route_workspace_bytes(T, kr, E) > STATIC_SCRATCH_BYTES
    nul = ctypes.c_void_p(0)
    st = lib.bsf_route_no_alloc(nul, T, kr, E, 0, 1, nul, nul, nul, nul, nul, T * kr, nul, nul, 0, 0, nul, nul,
                                0, nul)
    assert st == 3    # BSF_ERR_UNSUPPORTED, nothing enqueued


def test_no_alloc_route_rejects_assignment_count_overflow():
    """T * kr above INT32_MAX is refused before the product is formed."""
    require_gpu()
    lib = _lib.load()
    nul = ctypes.c_void_p(0)
    T, kr, E = 2**31, 8, 8
    assert lib.bsf_route_workspace_bytes(T, kr, E) == 0
    st = lib.bsf_route_no_alloc(nul, T, kr, E, 0, 1, nul, nul, nul, nul, nul, T * kr, nul, nul, 0, 0, nul, nul,
                                0, nul)
    assert st == 3    # BSF_ERR_UNSUPPORTED, nothing enqueued
