"""Pins for oracle.checks: closed forms of calc_diff = 1 - 2 sum(xy) / sum(x^2 + y^2)
(DeepGEMM article, "精度与吞吐的平衡点") and of the per-element bound."""

import numpy as np

from oracle import checks


def test_calc_diff_closed_forms():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(1000)
    assert checks.calc_diff(x, x) == 0.0
    assert abs(checks.calc_diff(x, -x) - 2.0) < 1e-15
    assert abs(checks.calc_diff(x, np.zeros_like(x)) - 1.0) < 1e-15
    for c in (0.5, 1.001, 3.0):
        assert abs(checks.calc_diff(x, c * x) - (1 - 2 * c / (1 + c * c))) < 1e-12
    # a 1e-3 relative perturbation on every element stays well inside the FP8 bound
    assert checks.calc_diff(x, x * (1 + 1e-3 * rng.standard_normal(1000))) < checks.CALC_DIFF_MAX


def test_elementwise_bound():
    ref = np.array([1.0, -2.0, 0.0, 1e-6])
    rms = np.sqrt(np.mean(ref ** 2))
    d = ref + np.array([2.0 ** -7, -2 * 2.0 ** -7, 1e-3 * rms, 0.0])
    assert checks.elementwise_ok(d, ref).all()
    d_bad = ref + np.array([2.0 ** -6, 0, 0, 0])
    assert list(checks.elementwise_ok(d_bad, ref)) == [False, True, True, True]
