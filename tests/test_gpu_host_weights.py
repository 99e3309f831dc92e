"""Host-resident weights ("AsymGEMM" README, "Asymmetric Memory Path"): the
grouped GEMM reads B and its scale factors from pinned host memory through
their device-mapped addresses.  The result must be bit-identical to the same
GEMM with the weights in HBM (the arithmetic is the same kernel's), and within
the oracle tolerance."""

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp8_route_gb300 import ops
from tests.gpu_util import bits16, check_expert_block, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def test_checksum_reads_device_and_host_memory(dev):
    g = torch.Generator().manual_seed(3)
    host = torch.randint(-2 ** 31, 2 ** 31 - 1, (1 << 18,), generator=g, dtype=torch.int64).pin_memory()
    ref = int(np.bitwise_xor.reduce(host.numpy().view(np.uint64)))
    on_dev = ops.checksum_u64(host.to(dev))
    via_link = ops.checksum_u64(host, host_mapped=True)
    torch.cuda.synchronize()
    assert int(on_dev.item()) & (2 ** 64 - 1) == ref
    assert int(via_link.item()) & (2 ** 64 - 1) == ref


def _problem(E, N, K, rows, seed, dev):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g) * 0.02).to(torch.bfloat16)
    aq, asf = ops.quantise_act(x.to(dev))
    bq, sf128 = ops.quantise_weight(w.to(dev))
    sfb = ops.prepare_weight_sf(sf128, K)
    return x, w, aq, asf, bq, sfb


@pytest.mark.parametrize("max_m,N", [(64, 384), (320, 384), (128, 512)])
def test_masked_host_weights_bitwise_equal_to_hbm_weights(dev, max_m, N):
    E, K = 6, 1024
    masked = np.minimum(np.array([0, 3, 17, 64, 200, max_m]), max_m)
    x, w, aq, asf, bq, sfb = _problem(E, N, K, E * max_m, max_m, dev)
    mm = torch.as_tensor(masked, dtype=torch.int32, device=dev)
    d_hbm = ops.grouped_gemm_masked(aq, asf, bq, sfb, mm, max_m)
    bq_h, sfb_h = bq.cpu().pin_memory(), sfb.cpu().pin_memory()
    d_host = ops.grouped_gemm_masked(aq, asf, bq_h, sfb_h, mm, max_m, flags=ops.B_HOST_MAPPED)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    a_ref, asf_ref = oracle.quantise.quantise_act(bits16(x))
    b_ref, bsf_ref = oracle.quantise.quantise_weight(bits16(w))
    for e in range(E):
        s, c = e * max_m, int(masked[e])
        if c == 0:
            continue
        assert torch.equal(d_host[s:s + c].view(torch.int16), d_hbm[s:s + c].view(torch.int16))
        ref = oracle.gemm.expert_gemm(a_ref[s:s + c], asf_ref[s:s + c], b_ref[e], bsf_ref[e])
        check_expert_block(bits16(d_host[s:s + c]), ref, f"host weights, expert {e}")


def test_contig_host_weights_bitwise_equal_to_hbm_weights(dev):
    E, N, K = 3, 256, 640
    counts = np.array([5, 300, 40])
    seg = np.concatenate([[0], np.cumsum(counts)])
    x, w, aq, asf, bq, sfb = _problem(E, N, K, int(seg[-1]), 9, dev)
    segt = torch.as_tensor(seg, dtype=torch.int32, device=dev)
    ct = torch.as_tensor(counts, dtype=torch.int32, device=dev)
    d_hbm = ops.grouped_gemm_contig(aq, asf, bq, sfb, segt, ct)
    d_host = ops.grouped_gemm_contig(aq, asf, bq.cpu().pin_memory(), sfb.cpu().pin_memory(), segt, ct,
                                     flags=ops.B_HOST_MAPPED)
    torch.cuda.synchronize()
    assert torch.equal(d_host.view(torch.int16), d_hbm.view(torch.int16))
