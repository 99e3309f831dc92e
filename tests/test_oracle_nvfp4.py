"""Pins for oracle.nvfp4 (NVFP4: E2M1 values, UE4M3 scales per 16 elements).

* The E2M1 table against the closed-form landmarks of the format definition;
  round trips, ties to even, saturation, and the encoder against a brute-force
  nearest-value search written here.
* The tensor exponent is the least one that keeps every block scale <= 448.
* Hand-computed blocks; exact scale equivariance under x -> x * 2**m with
  j -> j + m; every element code is the nearest value of its block grid.
* Nibble order and SF byte order on hand-made words.
* The GEMM against exact rational arithmetic; the DeepGEMM article's FP4 x FP4
  threshold (calc_diff <= 0.02 against the unquantised product) and its
  FP4 / FP8 equivalence (the FP4 GEMM equals the FP8 GEMM on the same values).
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import checks, formats, gemm, nvfp4, quantise
from tests.exact import exact_bf16_bits


def test_e2m1_table_closed_form():
    t = nvfp4.e2m1_decode_table()
    assert list(t[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(t[8:]) == [-v for v in t[:8]]
    assert np.signbit(t[8])


def test_e2m1_round_trip_every_code():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(nvfp4.e2m1_encode(nvfp4.e2m1_decode(codes)), codes)


def test_e2m1_ties_to_even_and_saturation():
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for y, want in ties.items():
        assert nvfp4.e2m1_decode(nvfp4.e2m1_encode(y)) == want, y
        assert nvfp4.e2m1_decode(nvfp4.e2m1_encode(-y)) == -want, y
    for y in (6.0, 6.5, 7.0, 100.0, np.inf):
        assert nvfp4.e2m1_encode(y) == 7 and nvfp4.e2m1_encode(-y) == 15
    assert nvfp4.e2m1_encode(-0.1) == 8                     # sign kept on a zero result


def test_e2m1_encoder_matches_brute_force_nearest():
    rng = np.random.default_rng(3)
    y = np.concatenate([rng.uniform(-7, 7, 20000), rng.standard_normal(20000)])
    vals = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = nvfp4.e2m1_decode(nvfp4.e2m1_encode(y))
    for v, g in zip(y, got):
        m = min(abs(v), 6.0)
        best = min(range(8), key=lambda c: (abs(m - vals[c]), c % 2))   # nearest, then even code
        assert abs(g) == vals[best] and (g == 0 or np.sign(g) == np.sign(v)), v


def test_global_exponent_is_least():
    rng = np.random.default_rng(4)
    amax = np.concatenate([np.exp2(rng.uniform(-60, 60, 50000)), [2688.0, 2688.0 * 2 ** -5, 1344.0001]])
    j = nvfp4.global_exponent(amax)
    assert np.all(amax <= 2688.0 * np.exp2(j.astype(float)))
    assert np.all(amax > 2688.0 * np.exp2(j.astype(float) - 1))
    assert nvfp4.global_exponent(0.0) == 0
    assert nvfp4.global_exponent(2688.0) == 0 and nvfp4.global_exponent(2688.5) == 1


def _block(vals):
    row = np.zeros(64)
    row[:len(vals)] = vals
    return formats.bf16_round(row[None, :])


def test_hand_computed_blocks():
    # amax 6 -> scale 1 (E4M3 code 0x38): values are their own codes
    q, sc = nvfp4.quantise_rows(_block([6.0, 3.0, -1.5, 0.25, 0.75, -4.0]), 0)
    assert sc[0, 0] == 0x38 and np.all(sc[0, 1:] == 0)
    codes = nvfp4.unpack_e2m1(q)[0, :6]
    assert list(nvfp4.e2m1_decode(codes)) == [6.0, 3.0, -1.5, 0.0, 1.0, -4.0]
    # amax 7 -> 7/6 = 1.1666 -> E4M3 1.125 (code 0x39); 7 / 1.125 = 6.2 saturates to 6
    q, sc = nvfp4.quantise_rows(_block([7.0, 1.0]), 0)
    assert sc[0, 0] == 0x39
    assert list(nvfp4.e2m1_decode(nvfp4.unpack_e2m1(q)[0, :2])) == [6.0, 1.0]   # 1 / 1.125 = 0.89 -> 1
    # tensor exponent j = 3: the same block with values x 8 gives the same codes
    q8, sc8 = nvfp4.quantise_rows(_block([56.0, 8.0]), 3)
    assert np.array_equal(q8, q) and np.array_equal(sc8, sc)
    # an all-zero block: scale code 0, element codes 0
    q, sc = nvfp4.quantise_rows(_block([]), 0)
    assert np.all(q == 0) and np.all(sc == 0)


def test_scale_equivariance():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 256)) * np.exp2(rng.integers(-8, 8, (16, 1)))
    xb = formats.bf16_round(x)
    q0, s0 = nvfp4.quantise_rows(xb, 0)
    for m in (-5, -1, 2, 7):
        qm, sm = nvfp4.quantise_rows(formats.bf16_round(formats.bf16_bits_to_f64(xb) * 2.0 ** m), m)
        assert np.array_equal(qm, q0) and np.array_equal(sm, s0), m


def test_every_element_is_a_nearest_grid_value():
    rng = np.random.default_rng(6)
    x = formats.bf16_round(rng.standard_normal((8, 512)) * 3)
    j = -2
    q, sc = nvfp4.quantise_rows(x, j)
    xv = formats.bf16_bits_to_f64(x)
    deq = nvfp4.dequant(q, sc, j)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    s = np.repeat(formats.e4m3_decode(sc), 16, axis=1) * 2.0 ** j
    for r in range(x.shape[0]):
        for k in range(x.shape[1]):
            cand = np.sign(xv[r, k]) * grid * s[r, k]
            best = np.min(np.abs(xv[r, k] - cand))
            assert abs(xv[r, k] - deq[r, k]) <= best * (1 + 2 ** -20) + 1e-300, (r, k)


def test_nibble_and_sf_byte_order():
    assert list(nvfp4.pack_e2m1(np.array([2, 4, 15, 1]))) == [0x42, 0x1F]     # 1.0, 2.0 | -6, 0.5
    assert np.array_equal(nvfp4.unpack_e2m1(np.array([0x42, 0x1F], dtype=np.uint8)), [2, 4, 15, 1])
    sc = np.arange(2 * 8, dtype=np.uint8).reshape(2, 8) + 0x30          # rows 0, 1; K = 128
    w = nvfp4.pack_sf(sc).view(np.uint32)
    assert w.shape == (2, 4)
    assert w[0, 0] == 0x33323130 and w[1, 0] == 0x37363534 and w[0, 1] == 0x3B3A3938
    assert np.all(w[:, 2:] == 0)
    assert np.array_equal(nvfp4.unpack_sf(nvfp4.pack_sf(sc), 2), sc)


def _problem(seed, E=2, N=32, K=128, rows=(2, 3)):
    rng = np.random.default_rng(seed)
    R = sum(rows)
    x = formats.bf16_round(rng.standard_normal((R, K)) * np.exp2(rng.integers(-3, 4, (R, 1))))
    w = formats.bf16_round(rng.standard_normal((E, N, K)) * 0.02)
    wj = nvfp4.global_exponent(np.abs(formats.bf16_bits_to_f64(w)).reshape(E, -1).max(axis=1))
    aq, _, asc = nvfp4.quantise_act(x, 1)
    bq, _, bsc = nvfp4.quantise_weight(w, wj)
    counts = np.array(rows)
    seg = np.concatenate([[0], np.cumsum(counts)])
    return x, w, (aq, asc, 1, bq, bsc, wj, seg, counts)


def test_gemm_exact_rational_brute_force():
    _, _, (aq, asc, aj, bq, bsc, bj, seg, counts) = _problem(7)
    d, valid = nvfp4.grouped_gemm(aq, asc, aj, bq, bsc, bj, seg, counts)
    E, N, K2 = bq.shape
    K = 2 * K2
    e2m1 = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    e4m3 = formats.e4m3_decode_table()

    def val(packed_row, sc_row, j, k):
        byte = int(packed_row[k // 2])
        code = (byte >> 4) if k % 2 else (byte & 0xF)
        v = e2m1[code & 7] * (-1 if code & 8 else 1)
        return v * Fraction(float(e4m3[sc_row[k // 16]])) * Fraction(2) ** int(j)

    for e in range(E):
        for r in range(seg[e], seg[e] + counts[e]):
            a = [val(aq[r], asc[r], aj, k) for k in range(K)]
            for n in range(0, N, 5):
                s = sum(a[k] * val(bq[e, n], bsc[e, n], bj[e], k) for k in range(K))
                assert int(d[r, n]) == exact_bf16_bits(Fraction(s)), (e, r, n)
    assert valid.sum() == counts.sum()


def test_fp4_by_fp4_within_the_pages_threshold():
    x, w, (aq, asc, aj, bq, bsc, bj, seg, counts) = _problem(8, E=2, N=128, K=1024, rows=(40, 24))
    d, _ = nvfp4.grouped_gemm(aq, asc, aj, bq, bsc, bj, seg, counts)
    xv, wv = formats.bf16_bits_to_f64(x), formats.bf16_bits_to_f64(w)
    for e in range(2):
        rows = slice(seg[e], seg[e] + counts[e])
        exact = xv[rows] @ wv[e].T
        diff = checks.calc_diff(formats.bf16_bits_to_f64(d[rows]), exact)
        assert diff <= 0.02, (e, diff)
        assert diff > 1e-4        # FP4 quantisation is visible: the check is not vacuous


def test_fp4_equals_fp8_on_the_same_values():
    rng = np.random.default_rng(9)
    R, E, N, K = 6, 2, 128, 256
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    xa = rng.choice(grid, (R, K)) * rng.choice([-1, 1], (R, K))
    xb = rng.choice(grid, (E, N, K)) * rng.choice([-1, 1], (E, N, K))
    xa[:, 0] = 6.0                      # every block reaches 6 somewhere -> scale 1
    xb[:, :, 0] = 6.0
    xa[:, ::16] = 6.0
    xb[:, :, ::16] = 6.0
    aq4, _, asc = nvfp4.quantise_act(formats.bf16_round(xa), 0)
    bq4, _, bsc = nvfp4.quantise_weight(formats.bf16_round(xb), np.zeros(E, dtype=np.int64))
    assert np.all(asc == 0x38) and np.all(bsc == 0x38)
    seg, counts = np.array([0, 4, 6]), np.array([4, 2])
    d4, _ = nvfp4.grouped_gemm(aq4, asc, 0, bq4, bsc, np.zeros(E), seg, counts)
    # the same values as FP8 with unit scales
    aq8 = formats.e4m3_encode(nvfp4.dequant(aq4, asc, 0))
    bq8 = formats.e4m3_encode(nvfp4.dequant(bq4.reshape(E * N, -1), bsc.reshape(E * N, -1), 0)).reshape(E, N, K)
    asf8 = np.full((R, K // 128), 127, dtype=np.uint8)
    bsf8 = np.ones((E, N // 128, K // 128), dtype=np.float32)
    d8, _ = gemm.grouped_gemm(aq8, asf8, bq8, bsf8, seg, counts)
    assert np.array_equal(d4, d8)
    assert checks.calc_diff(formats.bf16_bits_to_f64(d4), formats.bf16_bits_to_f64(d8)) < 1e-14


@pytest.mark.parametrize("j", [101, -101])
def test_tensor_exponent_limit(j):
    with pytest.raises(ValueError):
        nvfp4.quantise_rows(_block([1.0]), j)
