"""The pins catch plausible mistakes: each test plants one mistake in the oracle
(on the CPU, through monkeypatching) and checks that the corresponding pin
test fails.  Nothing here touches a GPU."""

import numpy as np
import pytest

from oracle import combine, formats, gemm, quantise, route
from tests import test_oracle_combine as pin_combine
from tests import test_oracle_formats as pin_formats
from tests import test_oracle_gemm as pin_gemm
from tests import test_oracle_quantise as pin_quantise
from tests import test_oracle_route as pin_route


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_ties_away_from_zero_is_caught(monkeypatch):
    orig = formats.e4m3_encode

    def ties_up(x):
        x = np.asarray(x, dtype=np.float64)
        return orig(np.nextafter(np.abs(x), np.inf) * np.sign(x) + 0.0 * x)   # nudges ties upwards

    monkeypatch.setattr(formats, "e4m3_encode", ties_up)
    _fails(pin_formats.test_e4m3_encode_ties_to_even)


def test_double_rounding_bf16_is_caught(monkeypatch):
    def via_float32(x):
        x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
        b = x32.view(np.uint32).astype(np.uint64)
        r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
        return r

    monkeypatch.setattr(formats, "bf16_round", via_float32)
    _fails(pin_formats.test_bf16_round_is_a_single_rounding)


def test_floor_instead_of_ceil_exponent_is_caught(monkeypatch):
    orig = quantise._block_exponent
    monkeypatch.setattr(quantise, "_block_exponent", lambda amax: orig(amax) - 1)
    _fails(pin_quantise.test_block_exponent_is_least_with_amax_bound)


def test_reversed_order_inside_expert_is_caught(monkeypatch, golden_dir):
    orig = np.argsort

    def unstable(a, kind=None, **kw):
        idx = orig(a, kind="stable", **kw)
        return idx[::-1][orig(np.asarray(a)[idx[::-1]], kind="stable")]   # same keys, reversed ties

    monkeypatch.setattr(route.np, "argsort", unstable)
    import json
    import os
    with open(os.path.join(golden_dir, "routing_example_t5_kr2_e4.json")) as f:
        ex = json.load(f)
    _fails(pin_route.test_worked_example_unaligned, ex)


def test_wrong_scale_block_index_is_caught(monkeypatch):
    def shifted(q, sf_bytes):
        v = formats.e4m3_decode(q)
        s = formats.ue8m0_to_scale(np.roll(sf_bytes, 1, axis=1))
        return v * np.repeat(s, quantise.BLOCK, axis=1)

    monkeypatch.setattr(gemm, "dequant_rows", shifted)
    _fails(pin_gemm.test_exact_rational_brute_force)


def test_wrong_weight_rows_are_caught(monkeypatch):
    orig = gemm.expert_gemm

    def reversed_rows(a_q, a_sf, b_q_e, b_sf_e):
        return orig(a_q, a_sf, b_q_e[::-1].copy(), b_sf_e[::-1].copy())   # output column n uses weight row N-1-n

    monkeypatch.setattr(gemm, "expert_gemm", reversed_rows)
    _fails(pin_gemm.test_exact_rational_brute_force)


def test_dropped_routing_weight_is_caught(monkeypatch, golden_dir):
    orig = combine.combine

    def unweighted(y_bits, output_index, topk_weights):
        return orig(y_bits, output_index, np.ones_like(np.asarray(topk_weights)))

    monkeypatch.setattr(combine, "combine", unweighted)
    _fails(pin_combine.test_page_formula_z0, golden_dir)


# ---------------------------------------------------------------- NVFP4
from oracle import nvfp4  # noqa: E402
from tests import test_oracle_nvfp4 as pin_nvfp4  # noqa: E402


def test_swapped_nibbles_are_caught(monkeypatch):
    orig = nvfp4.unpack_e2m1

    def swapped(packed):
        c = orig(packed)
        out = c.copy()
        out[..., 0::2], out[..., 1::2] = c[..., 1::2], c[..., 0::2]
        return out

    monkeypatch.setattr(nvfp4, "unpack_e2m1", swapped)
    # (a dot product is blind to the same swap on both operands; the byte-level pin is not)
    _fails(pin_nvfp4.test_nibble_and_sf_byte_order)


def test_e2m1_ties_away_from_zero_are_caught(monkeypatch):
    orig = nvfp4.e2m1_encode
    monkeypatch.setattr(nvfp4, "e2m1_encode", lambda y: orig(np.asarray(y, dtype=np.float64) * (1 + 2 ** -30)))
    _fails(pin_nvfp4.test_e2m1_ties_to_even_and_saturation)


def test_wrong_scale_divisor_is_caught(monkeypatch):
    monkeypatch.setattr(nvfp4, "quantise_rows", _scaled_divisor(nvfp4.quantise_rows))
    _fails(pin_nvfp4.test_hand_computed_blocks)


def _scaled_divisor(orig):
    def wrong(x_bits, j):
        # scales from amax / 4 instead of amax / 6: the same as quantising x * 1.5
        x = nvfp4.formats.bf16_bits_to_f64(x_bits) * 1.5
        return orig(nvfp4.formats.bf16_round(x), j)
    return wrong


def test_global_exponent_off_by_one_is_caught(monkeypatch):
    orig = nvfp4.global_exponent
    monkeypatch.setattr(nvfp4, "global_exponent", lambda a: orig(a) + 1)
    _fails(pin_nvfp4.test_global_exponent_is_least)


# ---------------------------------------------------------------- BF16
from oracle import bf16 as bf16_oracle  # noqa: E402
from tests import test_oracle_bf16 as pin_bf16  # noqa: E402


def test_bf16_wrong_expert_weights_are_caught(monkeypatch):
    orig = bf16_oracle.grouped_gemm
    monkeypatch.setattr(bf16_oracle, "grouped_gemm",
                        lambda a, b, seg, counts: orig(a, np.roll(b, 1, axis=0), seg, counts))
    _fails(pin_bf16.test_exact_rational_brute_force)


# ---------------------------------------------------------------- FP32 scale factors
from oracle import f32sf  # noqa: E402
from tests import test_oracle_f32sf as pin_f32sf  # noqa: E402


def test_f32sf_wrong_divisor_is_caught(monkeypatch):
    monkeypatch.setattr(f32sf, "_scale", lambda amax32: np.where(amax32 == 0, np.float32(1.0),
                                                                 amax32 / np.float32(224.0)).astype(np.float32))
    _fails(pin_f32sf.test_hand_computed_blocks)


def test_f32sf_dropped_weight_scale_is_caught(monkeypatch):
    orig = f32sf.grouped_gemm
    monkeypatch.setattr(f32sf, "grouped_gemm",
                        lambda aq, as_, bq, bs, seg, counts: orig(aq, as_, bq, np.ones_like(bs), seg, counts))
    _fails(pin_f32sf.test_gemm_exact_rational_brute_force)


# ---------------------------------------------------------------- routing, packing, block shape
def test_ignored_segment_alignment_is_caught(monkeypatch, golden_dir):
    orig = route.route

    def unaligned(topk_ids, num_experts, layout=route.CONTIGUOUS, align=1, max_m=0):
        return orig(topk_ids, num_experts, layout, 1, max_m)              # align dropped

    monkeypatch.setattr(route, "route", unaligned)
    import json
    import os
    with open(os.path.join(golden_dir, "routing_example_t5_kr2_e4.json")) as f:
        ex = json.load(f)
    _fails(pin_route.test_worked_example_aligned_128, ex)


def test_dropped_routes_counted_as_expert_zero_are_caught(monkeypatch):
    orig = route.route

    def drops_to_zero(topk_ids, num_experts, layout=route.CONTIGUOUS, align=1, max_m=0):
        ids = np.asarray(topk_ids).copy()
        ids[ids < 0] = 0                                                   # -1 routed to expert 0
        return orig(ids, num_experts, layout, align, max_m)

    monkeypatch.setattr(route, "route", drops_to_zero)
    _fails(pin_route.test_brute_force_small, 0)


def test_reversed_sf_byte_order_is_caught(monkeypatch):
    orig = quantise.pack_sf

    def big_endian(sf_bytes, ld=None):
        w = orig(sf_bytes, ld).view(np.uint32)
        return w.byteswap().view(np.int32)                                 # byte j <-> byte 3 - j

    monkeypatch.setattr(quantise, "pack_sf", big_endian)
    _fails(pin_quantise.test_pack_sf_byte_order_and_round_trip)


def test_weight_blocks_of_1x128_are_caught(monkeypatch):
    def rowwise(w_bf16_bits):
        w = np.asarray(w_bf16_bits)
        E, N, K = w.shape
        q, by = quantise.quantise_act(w.reshape(E * N, K))                # 1 x 128 blocks instead of 128 x 128
        s = np.ldexp(1.0, by.reshape(E, N, K // 128).astype(np.int64) - 127).astype(np.float32)
        return q.reshape(E, N, K), s[:, ::128, :]

    monkeypatch.setattr(quantise, "quantise_weight", rowwise)
    _fails(pin_quantise.test_weight_blocks_are_128x128)
