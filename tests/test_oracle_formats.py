"""Pins for oracle.formats: E4M3 decode/encode, UE8M0, BF16 rounding.

The E4M3 layout (1/4/3 bits, max 448) is the DeepGEMM article's ("FP8 的精度陷阱");
UE8M0 is its "补偿机制一".  Library routine used as the independent reference:
torch's CPU float8_e4m3fn and bfloat16 casts (both round to nearest even).
"""

import numpy as np
import pytest
import torch

from oracle import formats


def test_e4m3_decode_landmarks():
    t = formats.e4m3_decode_table()
    assert t[0x00] == 0.0
    assert t[0x01] == 2.0 ** -9          # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x38] == 1.0                # exponent field 7 = bias
    assert t[0x7E] == 448.0              # largest finite
    assert t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.sum(np.isnan(t)) == 2
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    pos = t[:127]
    assert np.all(np.diff(pos) > 0)      # magnitude increases with the code
    assert np.array_equal(t[0x80:0xFF], -t[:127])


def test_e4m3_decode_matches_torch_view():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = formats.e4m3_decode_table()
    same = (ref == mine) | (np.isnan(ref) & np.isnan(mine))
    assert same.all()


def test_e4m3_round_trip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = formats.e4m3_encode(formats.e4m3_decode(codes))
    assert np.array_equal(back, codes)


def _e4m3_torch(x32):
    return torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_random():
    rng = np.random.default_rng(7)
    n = 1_000_000
    mag = np.exp2(rng.uniform(-14, np.log2(448.0), n))
    x = (mag * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    assert np.array_equal(formats.e4m3_encode(x.astype(np.float64)), _e4m3_torch(x))


def test_e4m3_encode_ties_to_even():
    pos = formats.e4m3_decode_table()[:127]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)   # exact in float32
    x = np.concatenate([mids, -mids])
    mine = formats.e4m3_encode(x.astype(np.float64))
    assert np.array_equal(mine, _e4m3_torch(x))
    # every tie lands on the even code
    assert np.all(mine[: len(mids)] % 2 == 0)


def test_e4m3_encode_saturates_and_signed_zero():
    x = np.array([448.0, 460.0, 1e6, -1e6, -1e-30, 0.0, 2.0 ** -10, 2.0 ** -10 * 1.0001])
    c = formats.e4m3_encode(x)
    assert list(c) == [0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00, 0x00, 0x01]


def test_ue8m0_round_trip_and_pow2_check():
    b = np.arange(1, 255, dtype=np.uint8)
    s = formats.ue8m0_to_scale(b)
    assert np.array_equal(formats.scale_to_ue8m0(s), b)
    bits = np.array([0x3F800000, 0x00800000, 0x7F000000, 0x3F800001, 0xBF800000, 0x3FC00000],
                    dtype=np.uint32)
    assert list(formats.is_power_of_two_f32(bits)) == [True, True, True, False, False, False]
    with pytest.raises(ValueError):
        formats.scale_to_ue8m0(np.array([3.0]))


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(11)
    n = 1_000_000
    raw = rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32)
    x = raw.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3.38e38)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(formats.bf16_round(x.astype(np.float64)), ref)


def test_bf16_round_is_a_single_rounding():
    # 1 + 2**-8 is the midpoint between bf16 1.0 and 1 + 2**-7; a value just
    # above it must round up.  A float32 intermediate would drop the 2**-30
    # and then tie to the even neighbour 1.0.
    x = np.array([1 + 2.0 ** -8 + 2.0 ** -30, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8 + 2.0 ** -30)])
    assert list(formats.bf16_round(x)) == [0x3F81, 0x3F80, 0x3F82, 0xBF81]
    x32 = np.float32(x[0])
    assert torch.tensor(x32).to(torch.bfloat16).view(torch.int16).item() == 0x3F80


def test_bf16_round_specials():
    x = np.array([0.0, -0.0, 3.4e38, -3.4e38, float.fromhex("0x1.fep127"), 2.0 ** -133, 2.0 ** -134, np.inf])
    b = formats.bf16_round(x)
    assert list(b) == [0x0000, 0x8000, 0x7F80, 0xFF80, 0x7F7F, 0x0001, 0x0000, 0x7F80]
    assert np.isnan(formats.bf16_bits_to_f64(formats.bf16_round(np.array([np.nan])))[0])
