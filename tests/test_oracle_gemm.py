"""Pins for oracle.gemm.

* Exact rational arithmetic on small shapes: every dequantised value is an
  exact fraction; the dot products are summed exactly and rounded once to
  BF16 by an integer procedure written here, independent of oracle.formats.
* "GEMM 执行方式" §4.1: a grouped GEMM equals P independent single GEMMs,
  whatever the placement of the segments (checked under a permuted,
  padded placement with garbage in the padding rows).
* DeepGEMM article "补偿机制一": a power-of-two scale change is exact, so
  scaling every A scale by 2**j scales D by exactly 2**j.
"""

from fractions import Fraction

import numpy as np

from oracle import formats, gemm, quantise
from tests.exact import exact_bf16_bits as _exact_bf16_bits


def _small_problem(seed, E=3, N=128, K=256, rows_per_expert=(2, 0, 3)):
    rng = np.random.default_rng(seed)
    rows = sum(rows_per_expert)
    x = formats.bf16_round(rng.standard_normal((rows, K)) * np.exp2(rng.integers(-3, 4, (rows, 1))))
    w = formats.bf16_round(rng.standard_normal((E, N, K)) * 0.02)
    aq, asf = quantise.quantise_act(x)
    bq, bsf = quantise.quantise_weight(w)
    counts = np.array(rows_per_expert)
    seg = np.concatenate([[0], np.cumsum(counts)])
    return aq, asf, bq, bsf, seg, counts


def test_exact_rational_brute_force():
    aq, asf, bq, bsf, seg, counts = _small_problem(1)
    d, valid = gemm.grouped_gemm(aq, asf, bq, bsf, seg, counts)
    dec = formats.e4m3_decode_table()
    E, N, K = bq.shape
    for e in range(E):
        for r in range(seg[e], seg[e] + counts[e]):
            a = [Fraction(float(dec[aq[r, k]])) * Fraction(2) ** (int(asf[r, k // 128]) - 127)
                 for k in range(K)]
            for n in range(0, N, 9):
                s = Fraction(0)
                for k in range(K):
                    bv = Fraction(float(dec[bq[e, n, k]])) * Fraction(float(bsf[e, n // 128, k // 128]))
                    s += a[k] * bv
                assert int(d[r, n]) == _exact_bf16_bits(s), (e, r, n)
    assert valid.sum() == counts.sum()


def test_grouped_equals_independent_single_gemms_under_permuted_placement():
    aq, asf, bq, bsf, seg, counts = _small_problem(2, E=4, rows_per_expert=(3, 1, 0, 5))
    ref, _ = gemm.grouped_gemm(aq, asf, bq, bsf, seg, counts)
    # place the experts in reverse order, each segment padded to 8 rows filled with garbage
    rng = np.random.default_rng(0)
    order = [3, 2, 1, 0]
    new_start = np.zeros(5, dtype=np.int64)
    pos = 0
    for e in order:
        new_start[e] = pos
        pos += -(-counts[e] // 8) * 8
    aq2 = rng.integers(0, 256, (pos, aq.shape[1]), dtype=np.uint8)
    aq2[(aq2 & 0x7F) == 0x7F] = 0
    asf2 = rng.integers(100, 140, (pos, asf.shape[1]), dtype=np.uint8)
    for e in range(4):
        aq2[new_start[e]:new_start[e] + counts[e]] = aq[seg[e]:seg[e] + counts[e]]
        asf2[new_start[e]:new_start[e] + counts[e]] = asf[seg[e]:seg[e] + counts[e]]
    d2, valid2 = gemm.grouped_gemm(aq2, asf2, bq, bsf, new_start, counts)
    for e in range(4):
        c = counts[e]
        single = gemm.expert_gemm(aq[seg[e]:seg[e] + c], asf[seg[e]:seg[e] + c], bq[e], bsf[e])
        assert np.array_equal(d2[new_start[e]:new_start[e] + c], single)
        assert np.array_equal(ref[seg[e]:seg[e] + c], single)
    assert valid2.sum() == counts.sum()


def test_power_of_two_scale_is_exact():
    aq, asf, bq, bsf, seg, counts = _small_problem(3)
    d, valid = gemm.grouped_gemm(aq, asf, bq, bsf, seg, counts)
    d2, _ = gemm.grouped_gemm(aq, (asf.astype(int) + 5).astype(np.uint8), bq, bsf, seg, counts)
    v = formats.bf16_bits_to_f64(d[valid])
    v2 = formats.bf16_bits_to_f64(d2[valid])
    assert np.array_equal(v2, v * 32.0)


def test_sampled_columns_match_full_problem():
    aq, asf, bq, bsf, seg, counts = _small_problem(4, E=2, N=256, rows_per_expert=(4, 3))
    d, _ = gemm.grouped_gemm(aq, asf, bq, bsf, seg, counts)
    cols = np.array([0, 5, 127, 128, 200, 255])
    for e in range(2):
        s, c = seg[e], counts[e]
        part = gemm.gemm_rows_cols(aq[s:s + c], asf[s:s + c], bq[e], bsf[e], cols)
        assert np.array_equal(part, d[s:s + c][:, cols])
