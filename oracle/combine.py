"""Weighted combine (un-permute) of expert outputs.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition ("GEMM 执行方式" §4.4 and §4.6; "CuTeDSL bei Perplexity", MoE
dispatch/combine): z_t = sum_{r < k_r} p[t, r] * y_packed[output_index[t, r]],
skipping dropped routes (output_index = -1).  Sum in float64, in r order,
rounded once to BF16 (nearest-even; the rounding is a reading).

Pins: ``tests/test_oracle_combine.py`` (z_0 = 0.70 y[0] + 0.30 y[5] and
0.70 y[0] + 0.30 y[256] of §4.4 / §4.6 with basis-vector rows, brute force).
"""

import numpy as np

from . import formats


def combine(y_bf16_bits, output_index, topk_weights):
    """z bf16 bits [T, N] from y bf16 bits [rows, N], output_index [T, k_r], weights f32 [T, k_r]."""
    y = formats.bf16_bits_to_f64(y_bf16_bits)
    idx = np.asarray(output_index, dtype=np.int64)
    p = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    T, kr = idx.shape
    z = np.zeros((T, y.shape[1]), dtype=np.float64)
    for r in range(kr):
        ok = idx[:, r] >= 0
        z[ok] += p[ok, r:r + 1] * y[idx[ok, r]]
    return formats.bf16_round(z)
