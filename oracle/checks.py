"""Acceptance metrics used to compare a result with the oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

* calc_diff (DeepGEMM article, "精度与吞吐的平衡点": the similarity measure of
  DeepGEMM's tests, FP8 x FP8 bound 0.001): 1 - 2 sum(x y) / sum(x^2 + y^2),
  in float64.  It is 0 for identical inputs and 1 against an all-zero input.
* Per-element bound (stated with the workload): |d - ref| <= 2**-7 |ref|
  + 1e-3 * rms(ref), rms over the block being checked.

* Combined-output bound (a reading: the pages state no combine tolerance):
  the combine is linear, so the per-element GEMM bound propagates to
  |z - z_ref| <= sum_r p[t, r] (2**-7 |y_ref| + 1e-3 rms_e) + 2**-7 |z_ref|,
  the last term covering the final bf16 rounding of z.

Pins: ``tests/test_oracle_checks.py`` (closed forms: x vs x, x vs -x, x vs 0,
x vs c x; the combined bound on a hand-computed case).
"""

import numpy as np

CALC_DIFF_MAX = 1e-3
REL_TOL = 2.0 ** -7
RMS_TOL = 1e-3


def calc_diff(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    denom = np.sum(x * x + y * y)
    if denom == 0:
        return 0.0
    return float(1.0 - 2.0 * np.sum(x * y) / denom)


def elementwise_ok(d, ref):
    """Boolean mask of elements within |d - ref| <= 2**-7 |ref| + 1e-3 rms(ref)."""
    d = np.asarray(d, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    return np.abs(d - ref) <= REL_TOL * np.abs(ref) + RMS_TOL * rms


def combined_bound(z_ref, y_ref, output_index, topk_weights, row_rms):
    """Per-element bound on |z - z_ref| propagated from the GEMM bound (see module doc)."""
    zr = np.asarray(z_ref, dtype=np.float64)
    y = np.asarray(y_ref, dtype=np.float64)
    idx = np.asarray(output_index)
    p = np.asarray(topk_weights, dtype=np.float64)
    bound = REL_TOL * np.abs(zr)
    for r in range(idx.shape[1]):
        ok = idx[:, r] >= 0
        rows = idx[ok, r]
        bound[ok] += p[ok, r:r + 1] * (REL_TOL * np.abs(y[rows]) + RMS_TOL * np.asarray(row_rms)[rows][:, None])
    return bound


def expert_row_rms(y_ref, seg_start, counts):
    """rms of each expert's valid output block, broadcast to that expert's rows."""
    y = np.asarray(y_ref, dtype=np.float64)
    out = np.zeros(y.shape[0])
    for e in range(len(counts)):
        s, c = int(seg_start[e]), int(counts[e])
        if c:
            out[s:s + c] = np.sqrt(np.mean(y[s:s + c] ** 2))
    return out
