"""BF16 grouped GEMM: D_e = A_e B_e^T with bf16 operands, no quantisation.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition: "AsymGEMM" README, "BF16 Asymmetric GEMM" (m_grouped_bf16_asym_gemm_nt_contiguous /
_masked: a bf16 [M, K], b bf16 [G, N, K], d bf16 [M, N], the same contiguous and masked layouts as
the FP8 calls); "GEMM 执行方式" §4.1 / §4.4 (P independent problems, Y_e = X_e W_e^T).  The DeepGEMM
article ("精度与吞吐的平衡点") holds the BF16 path to calc_diff 1e-5.

Every bf16 value is exact in float64, so is every product (8 + 8 significant bits); the float64 sum
over K carries rounding far below the bf16 resolution and is rounded once to bf16, nearest even.

Pins: ``tests/test_oracle_bf16.py`` (exact rational arithmetic on small shapes; grouped == one
problem per expert under a permuted placement).
"""

import numpy as np

from . import formats


def grouped_gemm(a_bits, b_bits, seg_start, counts):
    """a bf16 bits [rows, K], b bf16 bits [E, N, K] -> (d bf16 bits [rows, N], valid bool [rows])."""
    rows = a_bits.shape[0]
    E, N, _ = b_bits.shape
    d = np.zeros((rows, N), dtype=np.uint16)
    valid = np.zeros(rows, dtype=bool)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        s = int(seg_start[e])
        a = formats.bf16_bits_to_f64(a_bits[s:s + c])
        b = formats.bf16_bits_to_f64(b_bits[e])
        d[s:s + c] = formats.bf16_round(a @ b.T)
        valid[s:s + c] = True
    return d, valid


def gemm_rows_cols(a_bits, b_bits_e, cols):
    """Selected output columns of one expert problem."""
    a = formats.bf16_bits_to_f64(a_bits)
    b = formats.bf16_bits_to_f64(b_bits_e[np.asarray(cols)])
    return formats.bf16_round(a @ b.T)
