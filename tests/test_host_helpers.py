"""Host-side helpers of the binding (no device calls): packed-operand capacity, scale-word
strides, buffer shapes per operand format, and the single-launch dispatch limits."""

import pytest

from block_scaled_fp8_route_gb300 import ops


def test_route_capacity_needs_no_device_sync():
    # contiguous: every assignment plus the worst-case alignment padding of every expert
    assert ops.route_capacity(4096, 8, 128, ops.CONTIGUOUS, 128) == 4096 * 8 + 128 * 127
    assert ops.route_capacity(64, 2, 8, ops.CONTIGUOUS, 1) == 128
    # masked: one slot of max_m rows per expert
    assert ops.route_capacity(128, 8, 128, ops.MASKED, 64) == 128 * 64


@pytest.mark.parametrize("rows,ld", [(1, 4), (4, 4), (5, 8), (1024, 1024), (1027, 1028)])
def test_sf_ld_rounds_rows_up_to_four(rows, ld):
    assert ops.sf_ld(rows) == ld


@pytest.mark.parametrize("K,words", [(128, 1), (512, 1), (640, 2), (4096, 8), (7168, 14)])
def test_sf_words_one_per_512_values(K, words):
    assert ops.sf_words(K) == words


@pytest.mark.parametrize("fmt,a_cols,sf_rows,sf_dtype", [
    ("fp8", 1024, 2, "int32"), ("nvfp4", 512, 16, "int32"), ("bf16", 1024, None, None),
    ("fp8_f32sf", 1024, 8, "float32")])
def test_route_buffers_per_format(fmt, a_cols, sf_rows, sf_dtype):
    b = ops.RouteBuffers(10, 2, 4, ops.CONTIGUOUS, 128, K=1024, device="cpu", fmt=fmt)
    assert b.m_cap == 20 + 4 * 127
    assert b.a_packed.shape == (b.m_cap, a_cols)
    assert b.token_of_row.numel() == b.m_cap and b.m_indices.numel() == b.m_cap
    assert b.output_index.shape == (10, 2) and b.seg_start.numel() == 5
    if sf_rows is None:
        assert b.sfa_packed is None
    else:
        assert b.sfa_packed.shape == (sf_rows, ops.sf_ld(b.m_cap))
        assert str(b.sfa_packed.dtype).endswith(sf_dtype)


def test_single_launch_dispatch_limits():
    assert ops.dispatch_supported(2048, 8, 256)            # 16384 assignments, 256 experts
    assert not ops.dispatch_supported(2049, 8, 256)
    assert not ops.dispatch_supported(16, 8, 257)
