"""Pins for oracle.bf16: exact rational arithmetic, and grouped == independent problems."""

from fractions import Fraction

import numpy as np

from oracle import bf16, formats
from tests.exact import exact_bf16_bits


def _problem(seed, E=3, N=24, K=96, rows=(2, 0, 3)):
    rng = np.random.default_rng(seed)
    R = sum(rows)
    a = formats.bf16_round(rng.standard_normal((R, K)) * np.exp2(rng.integers(-6, 7, (R, 1))))
    b = formats.bf16_round(rng.standard_normal((E, N, K)) * 0.02)
    counts = np.array(rows)
    return a, b, np.concatenate([[0], np.cumsum(counts)]), counts


def test_exact_rational_brute_force():
    a, b, seg, counts = _problem(1)
    d, valid = bf16.grouped_gemm(a, b, seg, counts)
    av, bv = formats.bf16_bits_to_f64(a), formats.bf16_bits_to_f64(b)
    for e in range(b.shape[0]):
        for r in range(seg[e], seg[e] + counts[e]):
            for n in range(0, b.shape[1], 5):
                s = sum(Fraction(float(av[r, k])) * Fraction(float(bv[e, n, k])) for k in range(a.shape[1]))
                assert int(d[r, n]) == exact_bf16_bits(s), (e, r, n)
    assert valid.sum() == counts.sum()


def test_grouped_equals_independent_problems_under_permuted_placement():
    a, b, seg, counts = _problem(2, E=4, rows=(3, 1, 0, 5))
    ref, _ = bf16.grouped_gemm(a, b, seg, counts)
    order = [2, 3, 0, 1]
    new_start = np.zeros(5, dtype=np.int64)
    pos = 0
    for e in order:
        new_start[e] = pos
        pos += 8
    a2 = np.full((pos, a.shape[1]), 0x7FC0, dtype=np.uint16)        # NaN garbage in the padding
    for e in range(4):
        a2[new_start[e]:new_start[e] + counts[e]] = a[seg[e]:seg[e] + counts[e]]
    d2, valid = bf16.grouped_gemm(a2, b, new_start, counts)
    for e in range(4):
        assert np.array_equal(d2[new_start[e]:new_start[e] + counts[e]], ref[seg[e]:seg[e] + counts[e]])
    assert valid.sum() == counts.sum()
