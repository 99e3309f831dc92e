"""Block quantisation to E4M3 with power-of-two (UE8M0) scales, and SF packing.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition (DeepGEMM article, "补偿机制一" and "FP8 的精度陷阱"; the recipe
(gran_m, gran_n, gran_k) = (1, 128, 128)): for every block of values
(1 x 128 along K for activations, 128 x 128 for weights)

* amax = max |x| over the block;
* the scale is 2**e with e the smallest integer such that amax <= 448 * 2**e,
  i.e. e = ceil(log2(amax / 448)); readings: an all-zero block takes e = 0,
  and e is clamped to [-126, 127], so the UE8M0 byte e + 127 lies in
  [1, 254] and 2**e is a normal float32 (the article's power-of-two check
  rejects the subnormal 2**-127); the clamp only bites for amax < 448 * 2**-126;
* q = E4M3(x * 2**-e), nearest-even (x * 2**-e is exact: a power-of-two scale
  only moves the exponent).

SF packing (article, "补偿机制一" / "补偿机制三"): four UE8M0 bytes per int32,
MN-major: word [i, r] holds the bytes of K-blocks 4i .. 4i+3 of row r, byte j
(little-endian, bits 8j..8j+7) for K-block 4i + j (the byte order is a
reading; the pages do not fix it).  Bytes past the last K-block are 127
(scale 1.0; they are never used).  The row stride of the packed tensor is
the row count rounded up to a multiple of 4 (16 bytes), the TMA-aligned
stride of the article.

Pins: ``tests/test_oracle_quantise.py`` (closed-form exponent bounds, scale
equivariance under x -> x * 2**j, all-zero blocks, hand-computed blocks, error
bound of half an E4M3 step, packing round trip).
"""

import numpy as np

from . import formats

BLOCK = 128


def _block_exponent(amax):
    """Smallest integer e with amax <= 448 * 2**e, clamped to [-126, 127]; 0 if amax == 0.

    With amax = m * 2**ex exactly (frexp, m in [0.5, 1)) and 448 = 0.875 * 2**9:
    amax <= 0.875 * 2**(9 + e)  <=>  e >= ex - 9 when m <= 0.875, and
    e >= ex - 8 when m > 0.875.
    """
    amax = np.asarray(amax, dtype=np.float64)
    m, ex = np.frexp(amax)
    e = ex.astype(np.int64) - 9 + (m > 0.875).astype(np.int64)
    e = np.where(amax == 0, 0, e)
    return np.clip(e, -126, 127)


def quantise_act(x_bf16_bits):
    """Quantise activations [T, K] (bf16 bit patterns) per 1 x 128 block.

    Returns (q uint8 [T, K], sf_bytes uint8 [T, K/128]).
    """
    x = formats.bf16_bits_to_f64(x_bf16_bits)
    T, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 128")
    xb = x.reshape(T, K // BLOCK, BLOCK)
    amax = np.max(np.abs(xb), axis=2)
    e = _block_exponent(amax)
    q = formats.e4m3_encode(np.ldexp(xb, -e[:, :, None]))
    return q.reshape(T, K), (e + 127).astype(np.uint8)


def quantise_weight(w_bf16_bits):
    """Quantise weights [E, N, K] (bf16 bit patterns) per 128 x 128 block.

    Returns (q uint8 [E, N, K], sf128 float32 [E, N/128, K/128]) with every
    sf128 entry an exact power of two.
    """
    w = formats.bf16_bits_to_f64(w_bf16_bits)
    E, N, K = w.shape
    if N % BLOCK or K % BLOCK:
        raise ValueError("N and K must be multiples of 128")
    wb = w.reshape(E, N // BLOCK, BLOCK, K // BLOCK, BLOCK)
    amax = np.max(np.abs(wb), axis=(2, 4))
    e = _block_exponent(amax)
    q = formats.e4m3_encode(np.ldexp(wb, -e[:, :, None, :, None]))
    return q.reshape(E, N, K), np.ldexp(1.0, e).astype(np.float32)


def sf_ld(rows):
    """Row stride (in int32 words) of a packed MN-major SF tensor: rows rounded up to 4."""
    return (rows + 3) // 4 * 4


def pack_sf(sf_bytes, ld=None):
    """Pack per-row SF bytes [rows, nkb] into MN-major int32 [ceil(nkb/4), ld]."""
    sf_bytes = np.asarray(sf_bytes, dtype=np.uint8)
    rows, nkb = sf_bytes.shape
    ld = sf_ld(rows) if ld is None else ld
    nw = (nkb + 3) // 4
    padded = np.full((rows, nw * 4), 127, dtype=np.uint32)
    padded[:, :nkb] = sf_bytes
    words = np.zeros((nw, ld), dtype=np.uint32)
    for j in range(4):
        words[:, :rows] |= padded[:, j::4].T << np.uint32(8 * j)
    return words.view(np.int32)


def unpack_sf(words, rows, nkb):
    """Inverse of ``pack_sf``: MN-major int32 [nw, ld] -> bytes [rows, nkb]."""
    w = np.asarray(words).view(np.uint32)
    out = np.empty((rows, nkb), dtype=np.uint8)
    for kb in range(nkb):
        out[:, kb] = (w[kb // 4, :rows] >> np.uint32(8 * (kb % 4))) & 0xFF
    return out


def prepare_weight_sf(sf128):
    """Weight SFs fp32 [E, N/128, K/128] -> per-row packed int32 [E, ceil(K/512), N].

    Each output row n carries the UE8M0 bytes of its 128-row block n // 128;
    raises if any scale is not an exact power of two (article "补偿机制一").
    """
    sf128 = np.asarray(sf128, dtype=np.float32)
    E, nb, nkb = sf128.shape
    if not np.all(formats.is_power_of_two_f32(sf128.view(np.uint32))):
        raise ValueError("weight scale factor is not a power of two")
    b = formats.scale_to_ue8m0(sf128.astype(np.float64))        # [E, nb, nkb]
    per_row = np.repeat(b, BLOCK, axis=1)                      # [E, N, nkb]
    return np.stack([pack_sf(per_row[e], ld=nb * BLOCK) for e in range(E)])
