"""Grouped GEMM D_e = A_e * dequant(B_e)^T over per-expert row segments.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition:

* "GEMM 执行方式" §4.1: a grouped GEMM is P independent single GEMMs;
  §4.4: for every non-empty expert e, Y_e = X_e W_e^T with W_e in R^{N x K};
  §4.6: row r of the packed operand uses the weights of the expert owning r,
  and rows never mix along K.
* "AsymGEMM" README, API reference: the NT contraction with a (data, scale)
  pair per operand, BF16 output; "Token Layout Protocols": contiguous
  segments or masked fixed-stride slices.
* DeepGEMM article, "补偿机制一": dequantisation multiplies each E4M3 value
  by its block's power-of-two scale, which is exact.

Here both operands are dequantised exactly to float64 (each value has at
most 4 significant bits), multiplied with one float64 matmul per expert (a
library primitive; every product is exact, the sum carries float64 rounding
only, far below the BF16 resolution) and rounded once to BF16, nearest-even.
Only rows [seg_start[e], seg_start[e] + counts[e]) are computed; padding rows
have no defined value (§4.6) and are reported as invalid.

Pins: ``tests/test_oracle_gemm.py`` (bit equality with exact rational
arithmetic on small shapes, grouped == independent single GEMMs under a
permuted segment placement, scale folding).
"""

import numpy as np

from . import formats
from .quantise import BLOCK


def dequant_rows(q, sf_bytes):
    """Exact dequantisation of rows [rows, K] with per-row 1 x 128 UE8M0 bytes [rows, K/128]."""
    v = formats.e4m3_decode(q)
    s = formats.ue8m0_to_scale(sf_bytes)
    return v * np.repeat(s, BLOCK, axis=1)


def dequant_weight(q_e, sf128_e):
    """Exact dequantisation of one expert's weights [N, K] with 128 x 128 fp32 scales."""
    v = formats.e4m3_decode(q_e)
    s = np.asarray(sf128_e, dtype=np.float64)
    return v * np.repeat(np.repeat(s, BLOCK, axis=0), BLOCK, axis=1)


def expert_gemm(a_q, a_sf_bytes, b_q_e, b_sf128_e):
    """One expert problem: BF16 bits of dequant(A) @ dequant(B_e)^T, [rows, N]."""
    a = dequant_rows(a_q, a_sf_bytes)
    b = dequant_weight(b_q_e, b_sf128_e)
    return formats.bf16_round(a @ b.T)


def grouped_gemm(a_q, a_sf_bytes, b_q, b_sf128, seg_start, counts):
    """Grouped GEMM over packed rows.

    a_q uint8 [rows, K], a_sf_bytes uint8 [rows, K/128], b_q uint8 [E, N, K],
    b_sf128 float32 [E, N/128, K/128], seg_start [E+1], counts [E].
    Returns (d bf16 bits uint16 [rows, N], valid bool [rows]).
    """
    rows = a_q.shape[0]
    E, N, _ = b_q.shape
    d = np.zeros((rows, N), dtype=np.uint16)
    valid = np.zeros(rows, dtype=bool)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        s = int(seg_start[e])
        d[s:s + c] = expert_gemm(a_q[s:s + c], a_sf_bytes[s:s + c], b_q[e], b_sf128[e])
        valid[s:s + c] = True
    return d, valid


def gemm_rows_cols(a_q, a_sf_bytes, b_q_e, b_sf128_e, cols):
    """Selected output columns of one expert problem (for sampled checks at large sizes)."""
    a = dequant_rows(a_q, a_sf_bytes)
    cols = np.asarray(cols)
    blocks = np.asarray(b_sf128_e, dtype=np.float64)[cols // BLOCK]      # [ncols, K/128]
    b = formats.e4m3_decode(b_q_e[cols]) * np.repeat(blocks, BLOCK, axis=1)
    return formats.bf16_round(a @ b.T)
