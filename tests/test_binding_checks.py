"""The binding refuses host tensors where the library needs device pointers (a kernel would
otherwise read or write through an address it cannot use).  CPU-only: every check fires before
any device call."""

import numpy as np
import pytest
import torch

from block_scaled_fp8_route_gb300 import ops


def test_quantisers_refuse_host_tensors():
    x = torch.zeros((4, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ops.quantise_act(x)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ops.quantise_weight(torch.zeros((1, 128, 128), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA tensor"):
        ops.tile_weights(torch.zeros((1, 128, 128), dtype=torch.uint8))


def test_gemm_refuses_host_operands():
    a = torch.zeros((8, 128), dtype=torch.uint8)
    sfa = torch.zeros((1, 8), dtype=torch.int32)
    b = torch.zeros((1, 128, 128), dtype=torch.uint8)
    sfb = torch.zeros((1, 1, 128), dtype=torch.int32)
    seg = torch.as_tensor(np.array([0, 8]), dtype=torch.int32)
    cnt = torch.as_tensor(np.array([8]), dtype=torch.int32)
    d = torch.zeros((8, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ops.grouped_gemm_contig(a, sfa, b, sfb, seg, cnt, d=d)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ops.grouped_gemm_bf16_contig(torch.zeros((8, 128), dtype=torch.bfloat16),
                                     torch.zeros((1, 128, 128), dtype=torch.bfloat16), seg, cnt, d=d)


def test_host_mapped_weights_must_be_pinned_host_tensors():
    b = torch.zeros((1, 128, 128), dtype=torch.uint8)          # pageable host memory
    with pytest.raises(ValueError, match="pinned host"):
        ops._wptr(b, ops.B_HOST_MAPPED)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ops._wptr(b, 0)
    assert ops._wptr(None, ops.B_HOST_MAPPED) is None
