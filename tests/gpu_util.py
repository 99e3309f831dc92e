"""Helpers for the GPU parity tests: tensor <-> numpy bit views, oracle runs of a
workload, and the per-expert tolerance check of the grouped GEMM."""

import numpy as np
import torch

import oracle


def bits16(t):
    """bf16 tensor -> uint16 numpy array of its bit patterns (on the CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint8)


def i32(t):
    return t.detach().cpu().contiguous().numpy().astype(np.int64)


def require_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from block_scaled_fp8_route_gb300 import build, _lib
    _lib.load(build.build())
    return torch.device("cuda:0")


def check_expert_block(d_gpu_bits, ref_bits, what):
    """calc_diff <= 1e-3 and the per-element bound on one expert's valid block."""
    d = oracle.formats.bf16_bits_to_f64(d_gpu_bits)
    ref = oracle.formats.bf16_bits_to_f64(ref_bits)
    assert np.all(np.isfinite(d)), f"{what}: non-finite output"
    diff = oracle.checks.calc_diff(d, ref)
    assert diff <= oracle.checks.CALC_DIFF_MAX, f"{what}: calc_diff {diff:.3e}"
    ok = oracle.checks.elementwise_ok(d, ref)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} elements outside the bound, e.g. "
                             + ", ".join(f"{tuple(b)}: {d[tuple(b)]} vs {ref[tuple(b)]}" for b in bad))
    return diff


def check_combined(z_gpu_bits, z_ref_bits, y_ref_bits, output_index, topk_weights, row_rms, what):
    """Combined output: calc_diff <= 1e-3 and the GEMM bound propagated through the combine."""
    z = oracle.formats.bf16_bits_to_f64(z_gpu_bits)
    zr = oracle.formats.bf16_bits_to_f64(z_ref_bits)
    y = oracle.formats.bf16_bits_to_f64(y_ref_bits)
    diff = oracle.checks.calc_diff(z, zr)
    assert diff <= oracle.checks.CALC_DIFF_MAX, f"{what}: calc_diff {diff:.3e}"
    bound = oracle.checks.combined_bound(zr, y, output_index, topk_weights, row_rms)
    bad = np.abs(z - zr) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside the propagated bound"
    return diff


def expert_row_rms(y_ref_bits, seg_start, counts):
    return oracle.checks.expert_row_rms(oracle.formats.bf16_bits_to_f64(y_ref_bits), seg_start, counts)


def oracle_packed_operand(aq, asf_bytes, token_of_row):
    """Oracle scatter of quantised token rows into packed rows (padding: zero data, byte 127)."""
    rows = oracle.route.scatter_rows(aq, token_of_row)
    sfb = oracle.route.scatter_rows(asf_bytes, token_of_row, pad_value=127)
    return rows, sfb


def check_combine_of_own_y(z_gpu_bits, y_gpu_bits, output_index, topk_weights, what):
    """The combine kernel alone: z from the GPU's own y against the float64 combine of that y.

    The kernel accumulates k_r products in FP32 and rounds once to bf16, so
    |z - z64| <= one bf16 step of z64 (2**-7 |z64|) + the FP32 summation error
    2 k_r 2**-24 sum_r |p_r y_r| (the factor 2 covers the final rounding of a
    sum that moved across a power of two).  Without cancellation the second
    term is far below the first; where the k_r terms cancel it is what remains.
    """
    z_own = oracle.combine.combine(y_gpu_bits, output_index, topk_weights)
    y = oracle.formats.bf16_bits_to_f64(y_gpu_bits)
    idx = np.asarray(output_index)
    p = np.abs(np.asarray(topk_weights, dtype=np.float32).astype(np.float64))
    mag = np.zeros((idx.shape[0], y.shape[1]))
    for r in range(idx.shape[1]):
        ok = idx[:, r] >= 0
        mag[ok] += p[ok, r:r + 1] * np.abs(y[idx[ok, r]])
    zo = oracle.formats.bf16_bits_to_f64(z_own)
    bound = np.abs(zo) * 2.0 ** -7 + 2.0 * idx.shape[1] * 2.0 ** -24 * mag + 1e-30
    d = np.abs(oracle.formats.bf16_bits_to_f64(z_gpu_bits) - zo)
    bad = d > bound
    if bad.any():
        t, n = np.unravel_index(np.argmax(d / bound), d.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements of the combine outside one bf16 step + FP32 "
                             f"summation error, worst [{t}, {n}]: |d| {d[t, n]:.3e}, bound {bound[t, n]:.3e}, "
                             f"z64 {zo[t, n]:.3e}, sum|p y| {mag[t, n]:.3e}")
