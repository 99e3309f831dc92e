"""Pins for oracle.f32sf (FP8 with float32 scale factors)."""

from fractions import Fraction

import numpy as np

from oracle import f32sf, formats, gemm, quantise
from tests.exact import exact_bf16_bits


def _row(vals, K=128):
    r = np.zeros(K)
    r[:len(vals)] = vals
    return formats.bf16_round(r[None, :])


def test_hand_computed_blocks():
    q, s = f32sf.quantise_act(_row([448.0, -1.0, 3.5]))
    assert s[0, 0] == 1.0 and list(formats.e4m3_decode(q[0, :3])) == [448.0, -1.0, 3.5]
    # amax 3: s = 3/448 (not a power of two); x / s = 448, -149.33 -> E4M3 -144 (step 16 at 128..256)
    q, s = f32sf.quantise_act(_row([3.0, -1.0]))
    assert s[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert list(formats.e4m3_decode(q[0, :2])) == [448.0, -144.0]
    q, s = f32sf.quantise_act(_row([]))
    assert s[0, 0] == 1.0 and np.all(q == 0)


def test_codes_are_nearest_to_the_scaled_values():
    rng = np.random.default_rng(1)
    x = formats.bf16_round(rng.standard_normal((16, 512)) * np.exp2(rng.integers(-9, 9, (16, 1))))
    q, s = f32sf.quantise_act(x)
    xv = formats.bf16_bits_to_f64(x)
    y = xv / np.repeat(s.astype(np.float64), 128, axis=1)
    table = formats.e4m3_decode_table()[:127]
    got = formats.e4m3_decode(q)
    for r in range(0, 16, 3):
        for k in range(0, 512, 7):
            best = np.min(np.abs(np.abs(y[r, k]) - table))
            assert abs(abs(got[r, k]) - abs(y[r, k])) <= best * (1 + 2 ** -20) + 1e-300
    assert np.max(np.abs(got)) <= 448.0


def test_weight_blocks_are_128_by_128():
    rng = np.random.default_rng(2)
    w = formats.bf16_round(rng.standard_normal((2, 256, 256)) * 0.02)
    q, s = f32sf.quantise_weight(w)
    assert s.shape == (2, 2, 2)
    wv = formats.bf16_bits_to_f64(w)
    for e in range(2):
        for i in range(2):
            for j in range(2):
                amax = np.abs(wv[e, 128 * i:128 * (i + 1), 128 * j:128 * (j + 1)]).max()
                assert s[e, i, j] == np.float32(np.float32(amax) / np.float32(448.0))


def test_gemm_exact_rational_brute_force():
    rng = np.random.default_rng(3)
    E, N, K, rows = 2, 128, 256, (2, 3)
    x = formats.bf16_round(rng.standard_normal((5, K)) * np.exp2(rng.integers(-3, 4, (5, 1))))
    w = formats.bf16_round(rng.standard_normal((E, N, K)) * 0.02)
    aq, as_ = f32sf.quantise_act(x)
    bq, bs = f32sf.quantise_weight(w)
    seg, counts = np.array([0, 2, 5]), np.array(rows)
    d, _ = f32sf.grouped_gemm(aq, as_, bq, bs, seg, counts)
    dec = formats.e4m3_decode_table()
    for e in range(E):
        for r in range(seg[e], seg[e] + counts[e]):
            for n in range(0, N, 11):
                acc = Fraction(0)
                for k in range(K):
                    acc += (Fraction(float(dec[aq[r, k]])) * Fraction(float(as_[r, k // 128])) *
                            Fraction(float(dec[bq[e, n, k]])) * Fraction(float(bs[e, n // 128, k // 128])))
                assert int(d[r, n]) == exact_bf16_bits(acc), (e, r, n)


def test_equals_the_ue8m0_gemm_when_scales_are_powers_of_two():
    rng = np.random.default_rng(4)
    x = formats.bf16_round(rng.standard_normal((6, 256)))
    w = formats.bf16_round(rng.standard_normal((2, 128, 256)) * 0.02)
    aq, asf = quantise.quantise_act(x)                  # UE8M0 quantisation: power-of-two scales
    bq, bsf = quantise.quantise_weight(w)
    seg, counts = np.array([0, 4, 6]), np.array([4, 2])
    d8, _ = gemm.grouped_gemm(aq, asf, bq, bsf, seg, counts)
    d32, _ = f32sf.grouped_gemm(aq, formats.ue8m0_to_scale(asf).astype(np.float32), bq, bsf, seg, counts)
    assert np.array_equal(d8, d32)
