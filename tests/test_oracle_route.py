"""Pins for oracle.route: the worked example of "GEMM 执行方式" §4.2-§4.6, the
assignment count invariant R = T k_r = sum_e M_e (§4.2), and brute force."""

import json
import os

import numpy as np
import pytest

from oracle import route


@pytest.fixture(scope="module")
def example(golden_dir):
    with open(os.path.join(golden_dir, "routing_example_t5_kr2_e4.json")) as f:
        return json.load(f)


def test_worked_example_unaligned(example):
    r = route.route(example["topk_ids"], example["E"], route.CONTIGUOUS, align=1)
    u = example["unaligned"]
    assert list(r["M"]) == example["M_e"]
    assert r["rows_used"] == u["M_packed"] == example["T"] * example["k_r"]
    assert list(r["m_indices"]) == u["m_indices"]
    assert r["output_index"].tolist() == u["output_index"]
    assert list(r["token_of_row"]) == u["x_packed_tokens"]
    x = np.array(example["x"])
    packed = route.scatter_rows(x, r["token_of_row"])
    assert np.array_equal(packed, x[u["x_packed_tokens"]])
    for e, toks in enumerate(example["expert_tokens"]):
        s, c = r["seg_start"][e], r["counts"][e]
        assert list(r["token_of_row"][s:s + c]) == toks


def test_worked_example_aligned_128(example):
    r = route.route(example["topk_ids"], example["E"], route.CONTIGUOUS, align=128)
    a = example["aligned_128"]
    assert r["rows_used"] == a["M_packed"] == 512
    assert [[int(r["seg_start"][e]), int(r["seg_start"][e + 1])] for e in range(4)] == a["segments"]
    expect_m = np.concatenate([np.full(n, e) for e, n in a["m_indices_runs"]])
    assert np.array_equal(r["m_indices"], expect_m)
    assert r["output_index"].tolist() == a["output_index"]
    valid = {int(k): v for k, v in a["valid_rows"].items()}
    for row in range(512):
        assert r["token_of_row"][row] == valid.get(row, -1)


def test_masked_layout_on_example(example):
    r = route.route(example["topk_ids"], example["E"], route.MASKED, max_m=2)
    # expert 0 and 2 receive 3 tokens each; with max_m = 2 the last (x4) is dropped
    assert list(r["counts"]) == [2, 2, 2, 2]
    assert r["dropped"] == 2
    assert r["output_index"].tolist() == [[0, 4], [2, 6], [1, 5], [3, 7], [-1, -1]]


def _brute(ids, E, layout, align, max_m):
    T, kr = ids.shape
    M = [sum(1 for t in range(T) for j in range(kr) if ids[t, j] == e) for e in range(E)]
    if layout == route.CONTIGUOUS:
        starts = [0]
        for e in range(E):
            starts.append(starts[-1] + -(-M[e] // align) * align)
        cap = M
    else:
        starts = [e * max_m for e in range(E + 1)]
        cap = [min(m, max_m) for m in M]
    out = -np.ones((T, kr), dtype=np.int64)
    for e in range(E):
        n = 0
        for t in range(T):
            for j in range(kr):
                if ids[t, j] == e:
                    if n < cap[e]:
                        out[t, j] = starts[e] + n
                    n += 1
    return M, starts, out


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_small(seed):
    rng = np.random.default_rng(seed)
    T, kr, E = rng.integers(1, 40), rng.integers(1, 5), rng.integers(1, 9)
    ids = rng.integers(-1, E, (T, kr))          # duplicates and dropped (-1) routes included
    for layout, align, max_m in [(route.CONTIGUOUS, 1, 0), (route.CONTIGUOUS, 4, 0),
                                 (route.CONTIGUOUS, 128, 0), (route.MASKED, 1, 3)]:
        r = route.route(ids, E, layout, align=align, max_m=max_m)
        M, starts, out = _brute(ids, E, layout, align, max_m)
        assert list(r["M"]) == M
        assert list(r["seg_start"]) == starts
        assert np.array_equal(r["output_index"], out)
        assert sum(M) == int(np.sum(ids >= 0))


def test_invariant_R_equals_sum_M():
    rng = np.random.default_rng(99)
    T, kr, E = 300, 8, 64
    ids = np.stack([rng.permutation(E)[:kr] for _ in range(T)])
    r = route.route(ids, E)
    assert int(r["M"].sum()) == T * kr == r["rows_used"]
    # every assignment has a distinct row, and the row's token is the assignment's token
    rows = r["output_index"].reshape(-1)
    assert len(set(rows.tolist())) == T * kr
    assert np.array_equal(r["token_of_row"][rows], np.repeat(np.arange(T), kr))


def test_out_of_range_expert_rejected():
    with pytest.raises(ValueError):
        route.route(np.array([[0, 4]]), 4)
