"""Number formats: FP8 E4M3, UE8M0 scale bytes and BF16 rounding.

TEST INFRASTRUCTURE ONLY (see the package docstring).

E4M3 is defined by the DeepGEMM article, section "FP8 的精度陷阱": 1 sign bit,
4 exponent bits, 3 mantissa bits, range about +-448.  The article does not
spell out special values; the reading taken here is the common "e4m3fn"
convention (exponent bias 7, subnormals m * 2**-9, no infinities, codes 0x7F
and 0xFF are NaN, largest finite magnitude 448 = code 0x7E).

UE8M0 (article section "补偿机制一"): an unsigned 8-bit exponent; byte b
encodes the scale 2**(b - 127), i.e. the float32 bit pattern with sign 0,
exponent b and mantissa 0.  Byte 0xFF is never produced.

Rounding readings (the pages state none): E4M3 encoding is round to nearest,
ties to even, saturating to +-448 ("satfinite"); BF16 output rounding is round
to nearest, ties to even, applied once to the exact (float64) value.

Pins: ``tests/test_oracle_formats.py`` checks the decode table against the
format definition's closed-form landmarks, the encoder against torch's CPU
float8_e4m3fn cast (a library routine) on a million values and on every tie,
exhaustive round trips, and the BF16 rounding against torch's float32->bfloat16
cast plus hand-made ties that a float32 intermediate would get wrong.
"""

import numpy as np

E4M3_MAX = 448.0
_BF16_MAX = float.fromhex("0x1.fep127")      # (2 - 2**-7) * 2**127
_BF16_MIN_QUANTUM_EXP = -133                 # smallest bf16 subnormal is 2**-133


def e4m3_decode_table():
    """Value of every E4M3 code 0..255 as float64 (NaN for 0x7F / 0xFF)."""
    table = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        man = code & 0x7
        if exp_field == 0xF and man == 0x7:
            table[code] = np.nan
        elif exp_field == 0:
            table[code] = sign * man * 2.0 ** -9          # subnormal: (m/8) * 2**(1-7)
        else:
            table[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp_field - 7)
    return table


_DECODE = e4m3_decode_table()
# non-negative finite magnitudes, indexed by code 0..126 (monotone in the code)
_POS_VALUES = _DECODE[:127].copy()


def e4m3_decode(codes):
    """Decode an array of uint8 E4M3 codes to float64."""
    return _DECODE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x):
    """Encode float64 values to E4M3 codes: nearest value, ties to even, saturating.

    The candidate codes are the two neighbours of |x| in the ordered list of
    non-negative finite E4M3 values; the closer one wins, and on an exact tie
    the code with an even mantissa (even code, since the mantissa is the low
    bits) wins.  Magnitudes at or beyond 448 saturate to 448.  The sign bit is
    copied from x, so negative values that round to zero give 0x80.
    """
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    out = np.empty(x.shape, dtype=np.uint8)
    sat = mag >= E4M3_MAX
    idx_lo = np.searchsorted(_POS_VALUES, mag, side="right") - 1
    idx_lo = np.clip(idx_lo, 0, 125)
    idx_hi = idx_lo + 1
    d_lo = mag - _POS_VALUES[idx_lo]
    d_hi = _POS_VALUES[idx_hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (idx_hi % 2 == 0))
    code = np.where(pick_hi, idx_hi, idx_lo)
    code = np.where(sat, 126, code)
    code = np.where(np.isnan(x), 127, code)
    out[...] = code.astype(np.uint8)
    out |= np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return out


def ue8m0_to_scale(b):
    """Scale 2**(b - 127) of UE8M0 bytes, as float64."""
    b = np.asarray(b, dtype=np.int64)
    return np.ldexp(1.0, b - 127)


def scale_to_ue8m0(s):
    """UE8M0 byte of exact power-of-two float scales (raises if one is not)."""
    s = np.asarray(s, dtype=np.float64)
    mant, ex = np.frexp(s)
    if np.any(mant != 0.5) or np.any(s <= 0):
        raise ValueError("scale factor is not a positive power of two")
    b = ex - 1 + 127
    if np.any((b < 0) | (b > 254)):
        raise ValueError("scale factor exponent outside UE8M0 range")
    return b.astype(np.uint8)


def is_power_of_two_f32(bits_u32):
    """Power-of-two check on float32 bit patterns: sign and mantissa bits are 0."""
    bits = np.asarray(bits_u32, dtype=np.uint32)
    return (bits & np.uint32(0x807FFFFF)) == 0


def bf16_bits_to_f64(bits):
    """BF16 bit patterns (uint16) to float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_round(x):
    """Round float64 values once to BF16 (nearest, ties to even); returns uint16 bits.

    |x| is split as m * 2**ex with m in [0.5, 1); the bf16 quantum at that
    magnitude is 2**(ex - 8) (8 significant bits), floored at the subnormal
    quantum 2**-133.  |x| / quantum is rounded to an integer with ties to even
    (numpy rint), which is exact in float64, then scaled back.  Results above
    the largest finite bf16 become infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    _, ex = np.frexp(mag)
    qexp = np.maximum(ex - 8, _BF16_MIN_QUANTUM_EXP)
    r = np.ldexp(np.rint(np.ldexp(mag, -qexp)), qexp)
    r = np.where(r > _BF16_MAX, np.inf, r)
    r = np.where(np.isnan(x), np.nan, r)
    r = np.where(np.signbit(x), -r, r)
    bits32 = r.astype(np.float32).view(np.uint32)   # r is exactly representable
    return (bits32 >> 16).astype(np.uint16)
