"""Host-side work accounting of bench.py, per operand format (no GPU): the algorithmic bytes of
each kernel follow from the data layouts, written out here independently."""

import numpy as np

import bench
import workloads as W


def _decode():
    w = W.WORKLOADS["decode"]
    counts = np.full(w.E, 8)              # 1024 routed rows, every expert active
    return w, counts, int(w.E * w.max_m)


def test_weight_bytes_per_format():
    N, K = 3072, 4096
    assert bench.weight_bytes(N, K, "fp8") == N * K + N * (K // 512) * 4          # per-row UE8M0 words
    assert bench.weight_bytes(N, K, "nvfp4") == N * K // 2 + N * K // 16          # E2M1 + one byte per 16
    assert bench.weight_bytes(N, K, "bf16") == 2 * N * K
    assert bench.weight_bytes(N, K, "fp8_f32sf") == N * K + (N // 128) * (K // 128) * 4


def test_decode_gemm_bytes():
    w, counts, placed = _decode()
    rows = int(counts.sum())
    for fmt, row_bytes in (("fp8", 4096 + 8 * 4), ("nvfp4", 2048 + 256), ("bf16", 8192), ("fp8_f32sf", 4096 + 32 * 4)):
        b, flops = bench.step_work(w, counts, placed, fused_dispatch=fmt in ("fp8", "nvfp4"), fmt=fmt)
        assert b["gemm"] == w.E * bench.weight_bytes(w.N, w.K, fmt) + rows * (row_bytes + 2 * w.N), fmt
        assert flops == 2.0 * rows * w.N * w.K
        assert b["combine"] == w.T * w.kr * w.N * 2 + w.T * w.N * 2 + w.T * w.kr * 8


def test_dispatch_versus_separate_quantise_and_route():
    w, counts, placed = _decode()
    fused, _ = bench.step_work(w, counts, placed, fused_dispatch=True)
    split, _ = bench.step_work(w, counts, placed, fused_dispatch=False)
    assert "dispatch" in fused and "quantise" not in fused
    assert {"quantise", "route"} <= set(split)
    # the single launch never writes (or re-reads) the token-major quantised copy
    assert fused["dispatch"] < split["quantise"] + split["route"]
    bf, _ = bench.step_work(w, counts, placed, fmt="bf16")
    assert "quantise" not in bf and "dispatch" not in bf


def test_two_gemm_step_counts_the_second_gemm():
    w = W.WORKLOADS["prefill"]
    counts = np.full(w.E, 256)
    b, flops = bench.step_work(w, counts, int(counts.sum()), fmt="fp8")
    assert {"gemm", "gemm2", "quantise2"} <= set(b)
    assert flops == 2.0 * counts.sum() * (w.N * w.K + w.N2 * w.K2)


def test_binding_roofline_picks_the_longer_bound():
    # 1 TFLOP and 1 GB in 1 ms: t_F = 1e12 / 2e15 = 0.5 ms, t_B = 1e9 / 2e12 = 0.5 ms -> equal; nudge each way
    r = bench.binding_roofline(1e12, 1.2e9, 1.0, 2000.0, 2000.0)
    assert r["bound"] == "hbm" and abs(r["achieved"] - 1200.0) < 1e-9 and abs(r["frac"] - 0.6) < 1e-12
    assert abs(r["tensor_frac"] - 0.5) < 1e-12 and abs(r["roofline_frac"] - 0.6) < 1e-12
    r = bench.binding_roofline(1.6e12, 1.0e9, 1.0, 2000.0, 2000.0)
    assert r["bound"] == "tensor" and abs(r["achieved"] - 1600.0) < 1e-9 and abs(r["frac"] - 0.8) < 1e-12
    assert abs(r["roofline_frac"] - 0.8) < 1e-12
