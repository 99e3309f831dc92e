"""Pins for oracle.quantise (DeepGEMM article, "补偿机制一" and "补偿机制三").

The scale of a block is 2**e with e the least integer such that amax <= 448 * 2**e.
Checked against that definition directly (exact float64 powers of two), against
hand-computed blocks, scale equivariance (power-of-two scaling is exact), and a
brute-force nearest-value search for every quantised element.
"""

import numpy as np
import pytest

from oracle import formats, quantise


def _bf16(x):
    return formats.bf16_round(np.asarray(x, dtype=np.float64))


def test_block_exponent_is_least_with_amax_bound():
    rng = np.random.default_rng(3)
    amax = formats.bf16_bits_to_f64(_bf16(np.exp2(rng.uniform(-100, 100, 200_000))))
    e = quantise._block_exponent(amax)
    assert np.all(amax <= 448.0 * np.ldexp(1.0, e))
    assert np.all(amax > 448.0 * np.ldexp(1.0, e - 1))


@pytest.mark.parametrize("amax,byte", [(448.0, 127), (450.0, 128), (1.0, 119), (224.0, 126),
                                       (0.875, 118), (0.0, 127), (2.0 ** 100, 219)])
def test_hand_computed_blocks(amax, byte):
    x = np.zeros((1, 128))
    x[0, 17] = -amax
    q, sf = quantise.quantise_act(_bf16(x))
    assert sf[0, 0] == byte
    if amax:
        # the extreme element lands in the top binade of E4M3: no waste, no saturation
        # (amax * 2**-e lies in (224, 448], and rounding can only reach 224 from above)
        v = abs(formats.e4m3_decode(q[0, 17]))
        assert 224.0 <= v <= 448.0
    else:
        assert not np.any(formats.e4m3_decode(q))   # -0.0 keeps its sign bit (0x80)


def test_hand_block_values_exact():
    # amax = 448 -> scale 1: every bf16 value that is also an E4M3 value is kept exactly
    x = np.zeros((1, 128))
    x[0, :4] = [448.0, -1.5, 0.013671875, 3.0]       # 0.013671875 = 7 * 2**-9
    q, sf = quantise.quantise_act(_bf16(x))
    assert sf[0, 0] == 127
    assert list(formats.e4m3_decode(q[0, :4])) == [448.0, -1.5, 0.013671875, 3.0]


def test_nearest_value_brute_force_and_scale_equivariance():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 512)) * np.exp2(rng.integers(-6, 6, (8, 1)))
    xb = _bf16(x)
    q, sf = quantise.quantise_act(xb)
    xv = formats.bf16_bits_to_f64(xb)
    scaled = xv * np.repeat(np.ldexp(1.0, 127 - sf.astype(np.int64)), 128, axis=1)
    table = formats.e4m3_decode_table()
    finite = table[~np.isnan(table)]
    best = np.min(np.abs(scaled[..., None] - finite[None, None, :]), axis=2)
    got = np.abs(scaled - formats.e4m3_decode(q))
    assert np.array_equal(got, best)
    for j in (-5, 3, 20):
        q2, sf2 = quantise.quantise_act(_bf16(xv * 2.0 ** j))
        assert np.array_equal(q2, q)
        assert np.array_equal(sf2.astype(int), sf.astype(int) + j)


def test_weight_blocks_are_128x128():
    w = np.full((1, 256, 256), 0.01)
    w[0, 130, 200] = 50.0                     # lives in block (1, 1)
    q, sf = quantise.quantise_weight(_bf16(w))
    assert sf.shape == (1, 2, 2)
    e = np.log2(sf[0].astype(np.float64))
    assert e[1, 1] == quantise._block_exponent(formats.bf16_bits_to_f64(_bf16([50.0])))[0]
    assert e[0, 0] == e[0, 1] == e[1, 0] == quantise._block_exponent(
        formats.bf16_bits_to_f64(_bf16([0.01])))[0]
    assert np.all(formats.is_power_of_two_f32(sf.view(np.uint32)))


def test_pack_sf_byte_order_and_round_trip():
    b = np.array([[1, 2, 3, 4, 5], [9, 8, 7, 6, 5]], dtype=np.uint8)
    w = quantise.pack_sf(b)
    assert w.shape == (2, 4)
    assert w.view(np.uint32)[0, 0] == 0x04030201
    assert w.view(np.uint32)[1, 0] == 0x7F7F7F05
    assert w.view(np.uint32)[0, 1] == 0x06070809
    assert np.array_equal(quantise.unpack_sf(w, 2, 5), b)


def test_prepare_weight_sf_rows_and_check():
    sf = np.ldexp(1.0, np.arange(-3, 3).reshape(1, 2, 3)).astype(np.float32)
    packed = quantise.prepare_weight_sf(sf)
    assert packed.shape == (1, 1, 256)
    u = packed.view(np.uint32)[0, 0]
    assert u[0] == u[127] == (124 | 125 << 8 | 126 << 16 | 127 << 24)
    assert u[128] == u[255] == (127 | 128 << 8 | 129 << 16 | 127 << 24)
    bad = sf.copy()
    bad[0, 0, 0] = 3.0
    with pytest.raises(ValueError):
        quantise.prepare_weight_sf(bad)
