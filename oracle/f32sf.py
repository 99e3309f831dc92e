"""FP8 E4M3 operands with float32 scale factors (the scales are not cast to UE8M0).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition: "AsymGEMM" README, notation: ``disable_ue8m0_cast`` keeps the scale factors in float32
instead of UE8M0; the FP8 grouped GEMMs take (data, scale) pairs with the (1, 128, 128) recipe.
DeepGEMM article, "补偿机制一": a float32 scale that is not a power of two is applied with rounding
(the UE8M0 path exists to avoid exactly that), and "补偿机制二": without block-scaled MMA hardware the
scales are applied in software.

Readings (the pages give the scale's type, not its value):

* per block (1 x 128 along K for activations, 128 x 128 for weights) s = float32(amax / 448), one
  float32 division rounded to nearest even; an all-zero block takes s = 1;
* q = E4M3(float32(x / s)), one float32 division then nearest-even E4M3 with saturation;
* D[r, n] = BF16(sum_k q_a s_a q_b s_b), the products exact in float64 and the sum in float64,
  rounded once.

Pins: ``tests/test_oracle_f32sf.py`` (hand-computed blocks, element codes nearest to x / s, exact
rational GEMM, equality with the UE8M0 GEMM when every scale is a power of two).
"""

import numpy as np

from . import formats

BLOCK = 128


def _scale(amax32):
    with np.errstate(divide="ignore", invalid="ignore"):
        s = (amax32 / np.float32(448.0)).astype(np.float32)
    return np.where(amax32 == 0, np.float32(1.0), s).astype(np.float32)


def _codes(x32, s32):
    y = (x32 / s32).astype(np.float32)
    return formats.e4m3_encode(y.astype(np.float64))


def quantise_act(x_bf16_bits):
    """[T, K] bf16 bits -> (q uint8 [T, K], s float32 [T, K/128])."""
    x = formats.bf16_bits_to_f64(x_bf16_bits).astype(np.float32)
    T, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 128")
    xb = x.reshape(T, K // BLOCK, BLOCK)
    s = _scale(np.abs(xb).max(axis=2))
    q = _codes(xb, s[:, :, None]).reshape(T, K)
    return q, s


def quantise_weight(w_bf16_bits):
    """[E, N, K] bf16 bits -> (q uint8 [E, N, K], s float32 [E, N/128, K/128])."""
    w = formats.bf16_bits_to_f64(w_bf16_bits).astype(np.float32)
    E, N, K = w.shape
    if N % BLOCK or K % BLOCK:
        raise ValueError("N and K must be multiples of 128")
    wb = w.reshape(E, N // BLOCK, BLOCK, K // BLOCK, BLOCK)
    s = _scale(np.abs(wb).max(axis=(2, 4)))
    q = _codes(wb, s[:, :, None, :, None]).reshape(E, N, K)
    return q, s


def sf_ld(rows):
    return (rows + 3) // 4 * 4


def pack_act_sf(s, ld=None):
    """float32 [T, K/128] -> MN-major float32 [K/128][ld] (ld = T rounded up to 4)."""
    T, nb = s.shape
    out = np.zeros((nb, sf_ld(T) if ld is None else ld), dtype=np.float32)
    out[:, :T] = s.T
    return out


def grouped_gemm(a_q, a_s, b_q, b_s, seg_start, counts):
    """a_q [rows, K], a_s float32 [rows, K/128], b_q [E, N, K], b_s float32 [E, N/128, K/128]."""
    rows = a_q.shape[0]
    E, N, _ = b_q.shape
    d = np.zeros((rows, N), dtype=np.uint16)
    valid = np.zeros(rows, dtype=bool)
    for e in range(E):
        c = int(counts[e])
        if c == 0:
            continue
        st = int(seg_start[e])
        a = formats.e4m3_decode(a_q[st:st + c]) * np.repeat(a_s[st:st + c].astype(np.float64), BLOCK, axis=1)
        sb = np.repeat(np.repeat(b_s[e].astype(np.float64), BLOCK, axis=0), BLOCK, axis=1)
        b = formats.e4m3_decode(b_q[e]) * sb
        d[st:st + c] = formats.bf16_round(a @ b.T)
        valid[st:st + c] = True
    return d, valid
