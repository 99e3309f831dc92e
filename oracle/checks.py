"""Acceptance metrics used to compare a result with the oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

* calc_diff (DeepGEMM article, "精度与吞吐的平衡点": the similarity measure of
  DeepGEMM's tests, FP8 x FP8 bound 0.001): 1 - 2 sum(x y) / sum(x^2 + y^2),
  in float64.  It is 0 for identical inputs and 1 against an all-zero input.
* Per-element bound (stated with the workload): |d - ref| <= 2**-7 |ref|
  + 1e-3 * rms(ref), rms over the block being checked.

Pins: ``tests/test_oracle_checks.py`` (closed forms: x vs x, x vs -x, x vs 0,
x vs c x).
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
