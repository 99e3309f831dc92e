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


def test_combined_bound_hand_case():
    # two tokens, k_r = 2; expert rows 0 and 1 (expert 0), row 2 (expert 1)
    y = np.array([[1.0, -2.0], [3.0, 0.0], [0.5, 0.5]])
    rms = checks.expert_row_rms(y, [0, 2, 3], [2, 1])
    assert np.allclose(rms, [np.sqrt(14 / 4), np.sqrt(14 / 4), 0.5])
    idx = np.array([[0, 2], [1, -1]])
    p = np.array([[0.75, 0.25], [1.0, 0.0]])
    z = np.array([[0.875, -1.375], [3.0, 0.0]])
    b = checks.combined_bound(z, y, idx, p, rms)
    r0 = np.sqrt(14 / 4)
    expect0 = (2.0 ** -7 * np.abs(z[0]) + 0.75 * (2.0 ** -7 * np.abs(y[0]) + 1e-3 * r0)
               + 0.25 * (2.0 ** -7 * np.abs(y[2]) + 1e-3 * 0.5))
    expect1 = 2.0 ** -7 * np.abs(z[1]) + 1.0 * (2.0 ** -7 * np.abs(y[1]) + 1e-3 * r0)
    assert np.allclose(b, np.stack([expect0, expect1]), rtol=0, atol=1e-15)
