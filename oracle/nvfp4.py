"""NVFP4 operands: E2M1 values, one UE4M3 scale per 16 elements, and the grouped GEMM on them.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition:

* "AsymGEMM" README, "Key Features" and "FP4 Asymmetric GEMM": the FP4 mode
  is NVFP4 — E2M1 data packed two elements per byte, scale factors in FP8
  E4M3; the grouped GEMM takes (data, scale) pairs like the FP8 one and
  writes BF16.
* "CuTeDSL bei Perplexity" (Blackwell support): the NVFP4 quantiser takes
  the absolute maximum over 16 elements, i.e. one scale per 16 values.
* DeepGEMM article, "精度与吞吐的平衡点": a GEMM with both operands in FP4
  stays within calc_diff 0.02 of the BF16 product, and an FP4 GEMM equals
  the FP8 GEMM on the same values converted to FP8.

Readings (the pages fix none of these):

* E2M1: 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; no
  infinities or NaN; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7,
  bit 3 the sign.  Encoding is round to nearest, ties to the even code,
  saturating at 6; the sign bit is copied, so negative values that round to
  zero give code 8.
* Packing: element 2i of a row in the low nibble of byte i, element 2i + 1
  in the high nibble.
* Scales: one per 16 consecutive elements along K (1 x 16 blocks for both
  operands), unsigned E4M3 (the positive codes 0x00..0x7E).
* A power-of-two tensor scale 2**j (one j per activation tensor, one per
  expert for the weights) extends the E4M3 range: scale code = E4M3(amax / 6
  / 2**j) with amax the block's absolute maximum; element code =
  E2M1(x / (scale * 2**j)); the value is e2m1 * scale * 2**j.  Every step
  is one float32 operation rounded to nearest even (amax / 6, the multiply
  by 2**-j, the division), exactly as a float32 kernel computes it; a block
  whose scale rounds to 0 stores code 0 for every element.  The tensor
  exponent that puts the largest block scale into (224, 448] is the least j
  with amax <= 6 * 448 * 2**j (``global_exponent``); j is limited to
  [-100, 100].
* SF packing, like the FP8 contract of the DeepGEMM article ("补偿机制三"):
  four scale bytes per int32, MN-major; word [w, r] holds the scales of
  elements 64w .. 64w+63 of row r, byte i (bits 8i..8i+7) for elements
  64w + 16i .. 64w + 16i + 15.  Activations: [K/64][ld], ld = rows rounded
  up to 4; weights: [E][K/64][N].
* GEMM: D[r, n] = BF16(sum_k value(A[r, k]) * value(B_e[n, k])) with the
  values above, summed in float64 (every product is exact: at most 2 + 4
  significant bits per factor) and rounded once, nearest even.

Pins: ``tests/test_oracle_nvfp4.py`` (the E2M1 table against its closed form,
ties and saturation, brute-force nearest values, the least tensor exponent,
hand-computed blocks, scale equivariance, nibble and SF byte order, exact
rational GEMM, the pages' 0.02 FP4 x FP4 threshold and the FP4 / FP8
equivalence).
"""

import numpy as np

from . import formats

E2M1_MAX = 6.0
SF_BLOCK = 16          # elements per scale
WORD_K = 64            # elements covered by one packed int32 SF word
E4M3_MAX = 448.0
J_LIMIT = 100


def e2m1_decode_table():
    """Value of every E2M1 code 0..15 as float64."""
    table = np.empty(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 0x8 else 1.0
        exp_field = (code >> 1) & 0x3
        man = code & 0x1
        if exp_field == 0:
            table[code] = sign * man * 0.5                  # subnormal: (m/2) * 2**(1-1)
        else:
            table[code] = sign * (1.0 + man / 2.0) * 2.0 ** (exp_field - 1)
    return table


_DECODE = e2m1_decode_table()
_POS = _DECODE[:8].copy()        # 0, 0.5, 1, 1.5, 2, 3, 4, 6 (monotone in the code)


def e2m1_decode(codes):
    return _DECODE[np.asarray(codes, dtype=np.uint8) & 0xF]


def e2m1_encode(y):
    """Nearest E2M1 code of float values (ties to the even code, saturating at 6, sign copied)."""
    y = np.asarray(y, dtype=np.float64)
    mag = np.abs(y)
    lo = np.clip(np.searchsorted(_POS, mag, side="right") - 1, 0, 6)
    hi = lo + 1
    d_lo = mag - _POS[lo]
    d_hi = _POS[hi] - mag
    code = np.where((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)), hi, lo)
    code = np.where(mag >= E2M1_MAX, 7, code)
    return (code | np.where(np.signbit(y), 0x8, 0)).astype(np.uint8)


def pack_e2m1(codes):
    """[..., K] codes -> [..., K/2] bytes (even element in the low nibble)."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed):
    """[..., K/2] bytes -> [..., K] codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def global_exponent(amax):
    """Least integer j with amax <= 6 * 448 * 2**j, limited to [-100, 100]; 0 when amax == 0.

    6 * 448 = 2688 = 0.65625 * 2**12; with amax = m * 2**ex (frexp, m in
    [0.5, 1)): amax <= 0.65625 * 2**(12 + j)  <=>  j >= ex - 12 when
    m <= 0.65625, and j >= ex - 11 otherwise.
    """
    amax = np.asarray(amax, dtype=np.float64)
    m, ex = np.frexp(amax)
    j = ex.astype(np.int64) - 12 + (m > 0.65625).astype(np.int64)
    j = np.where(amax == 0, 0, j)
    return np.clip(j, -J_LIMIT, J_LIMIT)


def _pow2_f32(j):
    return np.float32(2.0 ** int(j))


def quantise_rows(x_bf16_bits, j):
    """Rows [R, K] of bf16 bit patterns with tensor exponent j.

    Returns (packed uint8 [R, K/2], scale codes uint8 [R, K/16]).
    """
    x = formats.bf16_bits_to_f64(x_bf16_bits)
    R, K = x.shape
    if K % WORD_K:
        raise ValueError("K must be a multiple of 64")
    if abs(int(j)) > J_LIMIT:
        raise ValueError("tensor exponent outside [-100, 100]")
    x32 = x.astype(np.float32)                                       # exact (bf16 values)
    blocks = x32.reshape(R, K // SF_BLOCK, SF_BLOCK)
    amax = np.abs(blocks).max(axis=2)                                # exact
    with np.errstate(over="ignore"):
        s32 = (amax / np.float32(6.0)).astype(np.float32)            # float32 division
        s32 = (s32 * _pow2_f32(-j)).astype(np.float32)               # float32 multiply
    sc = formats.e4m3_encode(s32.astype(np.float64))
    s = formats.e4m3_decode(sc)                                      # scale values (>= 0)
    den = (s * 2.0 ** int(j)).astype(np.float32)                     # exact
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (blocks / den[:, :, None]).astype(np.float32)            # float32 division
    codes = e2m1_encode(y.astype(np.float64))
    codes = np.where((s == 0)[:, :, None], 0, codes).astype(np.uint8)
    return pack_e2m1(codes.reshape(R, K)), sc.astype(np.uint8)


def sf_ld(rows):
    return (rows + 3) // 4 * 4


def pack_sf(scale_codes, ld=None):
    """Scale codes [R, K/16] -> int32 words [K/64][ld] (MN-major, byte i = block 4w + i)."""
    sc = np.asarray(scale_codes, dtype=np.uint32)
    R, nb = sc.shape
    ld = sf_ld(R) if ld is None else ld
    words = np.zeros((nb // 4, ld), dtype=np.uint32)
    for i in range(4):
        words[:, :R] |= sc[:, i::4].T << np.uint32(8 * i)
    return words.view(np.int32)


def unpack_sf(words, rows):
    """int32 words [K/64][ld] -> scale codes [rows, K/16]."""
    w = np.asarray(words).view(np.uint32)[:, :rows]
    nw = w.shape[0]
    out = np.empty((rows, 4 * nw), dtype=np.uint8)
    for i in range(4):
        out[:, i::4] = ((w >> np.uint32(8 * i)) & np.uint32(0xFF)).T
    return out


def quantise_act(x_bf16_bits, j=0):
    """Activations [T, K] -> (packed uint8 [T, K/2], sf int32 [K/64][sf_ld(T)], scale codes [T, K/16])."""
    q, sc = quantise_rows(x_bf16_bits, j)
    return q, pack_sf(sc), sc


def quantise_weight(w_bf16_bits, j):
    """Weights [E, N, K] with one exponent per expert -> (packed [E, N, K/2], sfb int32 [E][K/64][N],
    scale codes [E, N, K/16])."""
    w = np.asarray(w_bf16_bits)
    E, N, K = w.shape
    q = np.empty((E, N, K // 2), dtype=np.uint8)
    sc = np.empty((E, N, K // SF_BLOCK), dtype=np.uint8)
    sfb = np.empty((E, K // WORD_K, N), dtype=np.int32)
    for e in range(E):
        q[e], sc[e] = quantise_rows(w[e], int(j[e]))
        sfb[e] = pack_sf(sc[e], ld=N)
    return q, sfb, sc


def dequant(packed, scale_codes, j):
    """Exact values [R, K] of packed E2M1 rows with their scale codes and tensor exponent."""
    v = e2m1_decode(unpack_e2m1(packed))
    s = formats.e4m3_decode(scale_codes)
    return v * np.repeat(s, SF_BLOCK, axis=-1) * 2.0 ** int(j)


def grouped_gemm(a_packed, a_sc, a_j, b_packed, b_sc, b_j, seg_start, counts):
    """Grouped GEMM over packed rows (segments as in oracle.gemm).

    a_packed [rows, K/2], a_sc [rows, K/16], a_j int; b_packed [E, N, K/2],
    b_sc [E, N, K/16], b_j [E].  Returns (d bf16 bits uint16 [rows, N], valid bool [rows]).
    """
    rows = a_packed.shape[0]
    E, N, _ = b_packed.shape
    d = np.zeros((rows, N), dtype=np.uint16)
    valid = np.zeros(rows, dtype=bool)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        s = int(seg_start[e])
        a = dequant(a_packed[s:s + c], a_sc[s:s + c], a_j)
        b = dequant(b_packed[e], b_sc[e], int(b_j[e]))
        d[s:s + c] = formats.bf16_round(a @ b.T)
        valid[s:s + c] = True
    return d, valid


def gemm_rows_cols(a_packed, a_sc, a_j, b_packed_e, b_sc_e, b_j_e, cols):
    """Selected output columns of one expert problem (sampled checks at large sizes)."""
    cols = np.asarray(cols)
    a = dequant(a_packed, a_sc, a_j)
    b = dequant(b_packed_e[cols], b_sc_e[cols], b_j_e)
    return formats.bf16_round(a @ b.T)
