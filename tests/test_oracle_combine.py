"""Pins for oracle.combine: the combine formulas of "GEMM 执行方式" §4.4 (unaligned,
z_0 = 0.70 y[0] + 0.30 y[5]) and §4.6 (aligned, z_0 = 0.70 y[0] + 0.30 y[256]),
checked with basis-vector expert outputs, and brute force in exact rationals."""

import json
import os
from fractions import Fraction

import numpy as np

from oracle import combine, formats, route
from tests.exact import exact_bf16_bits as _exact_bf16_bits


def _basis_rows(rows, n):
    y = np.zeros((rows, n))
    y[np.arange(rows), np.arange(rows)] = 1.0
    return formats.bf16_round(y)


def test_page_formula_z0(golden_dir):
    with open(os.path.join(golden_dir, "routing_example_t5_kr2_e4.json")) as f:
        ex = json.load(f)
    w = np.array(ex["topk_weights"], dtype=np.float32)
    for key, align in (("unaligned", 1), ("aligned_128", 128)):
        r = route.route(ex["topk_ids"], ex["E"], route.CONTIGUOUS, align=align)
        rows = r["rows_used"]
        z = formats.bf16_bits_to_f64(combine.combine(_basis_rows(rows, rows), r["output_index"], w))
        expect = np.zeros(rows)
        for coef, row in ex[key]["z0_terms"]:
            expect[row] = formats.bf16_bits_to_f64(formats.bf16_round(np.float32(coef)))
        assert np.array_equal(z[0], expect)


def test_brute_force_exact():
    rng = np.random.default_rng(8)
    T, kr, rows, N = 7, 3, 16, 12
    y = formats.bf16_round(rng.standard_normal((rows, N)))
    idx = rng.integers(-1, rows, (T, kr))
    p = rng.random((T, kr)).astype(np.float32)
    z = combine.combine(y, idx, p)
    yv = formats.bf16_bits_to_f64(y)
    for t in range(T):
        for n in range(N):
            s = sum((Fraction(float(p[t, j])) * Fraction(float(yv[idx[t, j], n]))
                     for j in range(kr) if idx[t, j] >= 0), Fraction(0))
            assert int(z[t, n]) == _exact_bf16_bits(s) or (s == 0 and int(z[t, n]) in (0, 0x8000))
