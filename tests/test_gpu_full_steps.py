"""Whole-step parity at the full prefill and large sizes, in the configuration the
bench times.

The step is ``MoEPath.step`` with tiled weights (``BSF_B_TILED``) and both
GEMMs: quantise -> multi-block route (count / scan / assign, then fill) ->
gate-up grouped GEMM (the 256-row work items) -> quantise of the down input ->
down grouped GEMM -> combine.  It is compared with the oracle, which shares no
code with it and starts from the same bf16 inputs:

* routing arrays (counts, seg_start, output_index, token_of_row, m_indices)
  bit for bit ("GEMM 执行方式" §4.3 / §4.6);
* the packed operand rows and their scale bytes of every sampled expert, byte
  for byte (the quantiser and the scatter);
* both GEMMs on at least 8 experts each — the two smallest, the two largest,
  the experts holding most of the large batch's x50 outlier rows, and random
  ones — under the per-expert tolerance (calc_diff <= 1e-3 and
  |d - ref| <= 2**-7 |ref| + 1e-3 rms(ref));
* the combined output on 256 sampled tokens (the outlier tokens among them) on
  two 128-column blocks of the down projection, under the bound propagated
  from the GEMM tolerance (rms per expert over its sampled rows and columns),
  and on every column within one bf16 step (plus the FP32 summation error
  bound) of the float64 combine of the GPU's own y.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from block_scaled_fp8_route_gb300 import MoEPath, ops
from tests.gpu_util import (bits16, check_combine_of_own_y, check_combined, check_expert_block, i32,
                            require_gpu, u8)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _sampled_experts(counts, must, rng, n_random):
    active = [e for e in range(len(counts)) if counts[e] > 0]
    by_size = sorted(active, key=lambda e: (counts[e], e))
    pick = set(by_size[:2]) | set(by_size[-2:]) | set(must)
    rest = [e for e in active if e not in pick]
    pick |= set(rng.choice(rest, size=n_random, replace=False).tolist())
    return sorted(int(e) for e in pick)


def _expert_weights(w, dev, e, second):
    """Oracle quantisation of one expert's bf16 weights (regenerated from its own stream)."""
    N, K, tag = (w.N2, w.K2, 1) if second else (w.N, w.K, 0)
    wt = W.weights(w, device=dev, N=N, K=K, experts=[int(e)], tag=tag).cpu()
    bq, bsf = oracle.quantise.quantise_weight(bits16(wt))
    return bq[0], bsf[0]


@pytest.mark.parametrize("name", ["prefill", "large"])
def test_full_step_matches_oracle(dev, name):
    w = W.WORKLOADS[name]
    rng = np.random.default_rng(7)
    ids, p = W.routing(w)
    x = W.activations(w, device=dev)
    wt = W.weights(w, device=dev)
    wt2 = W.weights(w, device=dev, N=w.N2, K=w.K2, tag=1)
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=w.align, w2_bf16=wt2,
                   device=dev, expected_m=w.T * w.kr // w.E)
    del wt, wt2
    torch.cuda.empty_cache()
    h2 = W.activations(W.with_tokens(w, path.bufs.m_cap), device=dev, K=w.K2, tag=1)
    # the bench's configuration: tiled weights, split quantise + multi-block route
    assert path.flags & ops.B_TILED and not path.fused_dispatch
    assert w.T * w.kr > ops.DISPATCH_MAX_ASSIGNMENTS
    z = path.step(x, ids.to(dev), p.to(dev), h2)
    torch.cuda.synchronize()
    assert ops.device_error() == 0

    # ---- routing, bit for bit
    r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align)
    b = path.bufs
    used = r["rows_used"]
    counts, seg = r["counts"], r["seg_start"]
    assert np.array_equal(i32(b.counts), counts)
    assert np.array_equal(i32(b.seg_start), seg)
    assert np.array_equal(i32(b.output_index), r["output_index"])
    assert np.array_equal(i32(b.token_of_row)[:used], r["token_of_row"])
    assert np.array_equal(i32(b.m_indices)[:used], r["m_indices"])

    # ---- sampled experts: packed operand bytes and both GEMMs
    x_cpu = x.cpu()
    h2_cpu = h2.cpu()
    outlier_tok = np.nonzero(x_cpu.float().abs().amax(dim=1).numpy() > 20.0)[0]
    must = []
    if w.outlier_frac > 0:
        assert len(outlier_tok) == round(w.outlier_frac * w.T)
        hold = np.bincount(ids.numpy()[outlier_tok].reshape(-1), minlength=w.E)
        must = [int(e) for e in np.argsort(-hold, kind="stable")[:2]]
        assert all(hold[e] > 0 for e in must)
    experts = _sampled_experts(counts, must, rng, n_random=4)
    assert len(experts) >= 8
    sfa_words = b.sfa_packed.cpu().numpy()
    yg, y2g = bits16(path.y), bits16(path.y2)
    for e in experts:
        s, c = int(seg[e]), int(counts[e])
        toks = r["token_of_row"][s:s + c]
        a_ref, asf_ref = oracle.quantise.quantise_act(bits16(x_cpu[torch.as_tensor(toks)]))
        assert np.array_equal(u8(b.a_packed[s:s + c]), a_ref), f"{name} expert {e}: packed rows"
        assert np.array_equal(oracle.quantise.unpack_sf(sfa_words[:, s:s + c], c, w.K // 128), asf_ref), \
            f"{name} expert {e}: packed scale bytes"
        bq, bsf = _expert_weights(w, dev, e, second=False)
        check_expert_block(yg[s:s + c], oracle.gemm.expert_gemm(a_ref, asf_ref, bq, bsf),
                           f"{name} gate-up expert {e} ({c} rows)")
        a2, a2sf = oracle.quantise.quantise_act(bits16(h2_cpu[s:s + c]))
        bq2, bsf2 = _expert_weights(w, dev, e, second=True)
        check_expert_block(y2g[s:s + c], oracle.gemm.expert_gemm(a2, a2sf, bq2, bsf2),
                           f"{name} down expert {e} ({c} rows)")

    # ---- combined output on sampled tokens
    n_tok = 256
    extra = outlier_tok[:32]
    others = np.setdiff1d(np.arange(w.T), extra)
    toks = np.sort(np.concatenate([extra, rng.choice(others, n_tok - len(extra), replace=False)]))
    idx = r["output_index"][toks]                        # packed rows feeding the sampled tokens
    rows = np.unique(idx[idx >= 0])
    compact = np.full(idx.shape, -1, dtype=np.int64)
    compact[idx >= 0] = np.searchsorted(rows, idx[idx >= 0])
    cb = [0, w.N2 // 128 - 1]                            # first and last 128-column blocks
    cols = np.concatenate([np.arange(c * 128, (c + 1) * 128) for c in cb])
    owner = r["m_indices"][rows]
    y_ref = np.zeros((len(rows), len(cols)), dtype=np.uint16)
    a2_all, a2sf_all = oracle.quantise.quantise_act(bits16(h2_cpu[torch.as_tensor(rows)]))
    for e in np.unique(owner):
        sel = np.nonzero(owner == e)[0]
        wt2_e = W.weights(w, device=dev, N=w.N2, K=w.K2, experts=[int(e)], tag=1)
        wt2_e = wt2_e[:, torch.as_tensor(cols, device=dev)].cpu()
        bq2, bsf2 = oracle.quantise.quantise_weight(bits16(wt2_e))     # 128-row blocks stay whole
        y_ref[sel] = oracle.gemm.expert_gemm(a2_all[sel], a2sf_all[sel], bq2[0], bsf2[0])
    y_ref_f = oracle.formats.bf16_bits_to_f64(y_ref)
    row_rms = np.zeros(len(rows))
    for e in np.unique(owner):
        sel = owner == e
        row_rms[sel] = np.sqrt(np.mean(y_ref_f[sel] ** 2))
    pt = p.numpy()[toks]
    z_ref = oracle.combine.combine(y_ref, compact, pt)
    zg = bits16(z)[toks]
    check_combined(zg[:, cols], z_ref, y_ref, compact, pt, row_rms, f"{name} combined output")
    # the combine kernel alone, on every column: against the float64 combine of the GPU's own y2
    check_combine_of_own_y(zg, y2g[rows], compact, pt, f"{name} combine")
