"""Seeded synthetic MoE workloads shared by the tests, the smoke check and the bench.

This module only draws random inputs (bf16 activations and weights, top-k
expert ids and routing weights) with the shapes and distributions of the five
workloads; it holds none of the quantisation, routing, GEMM or combine
arithmetic.  Both the CUDA path and the CPU oracle consume the tensors it
returns.  Generation uses torch generators, on the CPU or on a CUDA device
(the two give different streams; a check always feeds the same tensors to
both sides).

Workloads (token count T, top-k_r of E experts, hidden K, expert width N):

* tiny:    T=64,   top-2 of 8,    K=N=256, contiguous (align 1 or 128)
* decode:  T=128,  top-8 of 128,  K=4096, N=3072, masked, max_m=64
* prefill: T=4096, top-8 of 128,  gate-up K=4096 N=3072, down K=1536 N=4096,
           Zipf-skewed experts, contiguous align 128
* large:   T=8192, top-8 of 256,  gate-up K=7168 N=4096, down K=2048 N=7168,
           8 experts empty, 1% outlier rows x50, contiguous align 128
* host:    decode shapes with weights in pinned host memory, T swept 16..4096

Distributions: activations N(0,1) drawn in float32 and rounded to bf16;
weights N(0, 0.02) drawn in float32 and rounded to bf16; top-k ids are k_r
distinct experts per token (a real top-k never repeats an expert): uniform
draws use the first k_r entries of a random permutation, skewed draws use
Gumbel-top-k on logits alpha * (-s * ln(rank + 1)) over a random ranking of
the experts (s = 1.1, alpha = 0.6, which gives per-expert counts of about 90
to 2000 at T=4096); routing weights are a softmax over k_r N(0,1) logits,
float32.
"""

from dataclasses import dataclass, field
from typing import Optional

import torch

CONTIGUOUS = 0
MASKED = 1


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    kr: int
    E: int
    K: int
    N: int
    layout: int
    align: int = 1
    max_m: int = 0
    K2: int = 0            # down-projection K (0: no second GEMM)
    N2: int = 0
    routing: str = "uniform"
    empty_experts: int = 0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    weights_on_host: bool = False
    seed: int = 1000
    notes: str = field(default="", compare=False)


WORKLOADS = {
    "tiny": Workload("tiny", T=64, kr=2, E=8, K=256, N=256, layout=CONTIGUOUS, align=1, seed=1000),
    "tiny_a128": Workload("tiny_a128", T=64, kr=2, E=8, K=256, N=256, layout=CONTIGUOUS, align=128, seed=1000),
    "decode": Workload("decode", T=128, kr=8, E=128, K=4096, N=3072, layout=MASKED, max_m=64, seed=1001),
    "prefill": Workload("prefill", T=4096, kr=8, E=128, K=4096, N=3072, layout=CONTIGUOUS, align=128,
                        K2=1536, N2=4096, routing="zipf", seed=1002),
    "large": Workload("large", T=8192, kr=8, E=256, K=7168, N=4096, layout=CONTIGUOUS, align=128,
                      K2=2048, N2=7168, empty_experts=8, outlier_frac=0.01, outlier_scale=50.0, seed=1003),
    "host": Workload("host", T=128, kr=8, E=128, K=4096, N=3072, layout=MASKED, max_m=64,
                     weights_on_host=True, seed=1004),
}

ZIPF_S = 1.1
ZIPF_ALPHA = 0.6


def with_tokens(w: Workload, T: int) -> Workload:
    d = dict(w.__dict__)
    d["T"] = T
    return Workload(**d)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def activations(w: Workload, device="cpu", K: Optional[int] = None, tag: int = 0):
    """bf16 [T, K] N(0,1) activations (outlier rows scaled before the bf16 rounding)."""
    K = w.K if K is None else K
    g = _gen(device, w.seed * 16 + 1 + tag)
    x = torch.randn(w.T, K, generator=g, device=device, dtype=torch.float32)
    if w.outlier_frac > 0:
        n_out = round(w.outlier_frac * w.T)
        rows = torch.randperm(w.T, generator=g, device=device)[:n_out]
        x[rows] *= w.outlier_scale
    return x.to(torch.bfloat16)


def weights(w: Workload, device="cpu", N: Optional[int] = None, K: Optional[int] = None,
            experts=None, tag: int = 0):
    """bf16 [E, N, K] N(0, 0.02) weights; ``experts`` selects a subset (same values per expert)."""
    N = w.N if N is None else N
    K = w.K if K is None else K
    ids = range(w.E) if experts is None else experts
    out = torch.empty(len(ids), N, K, dtype=torch.bfloat16, device=device)
    for i, e in enumerate(ids):
        g = _gen(device, (w.seed * 16 + 2 + tag) * 4096 + e)
        out[i] = (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    return out


def routing(w: Workload, device="cpu"):
    """(topk_ids int32 [T, k_r], topk_weights float32 [T, k_r]) on ``device``."""
    g = _gen("cpu", w.seed * 16 + 3)
    T, E, kr = w.T, w.E, w.kr
    if w.routing == "zipf":
        rank_of_expert = torch.randperm(E, generator=g)
        logits = ZIPF_ALPHA * (-ZIPF_S * torch.log(rank_of_expert.to(torch.float64) + 1.0))
        u = torch.rand(T, E, generator=g, dtype=torch.float64).clamp_min(1e-300)
        gumbel = -torch.log(-torch.log(u))
        ids = torch.topk(logits[None, :] + gumbel, kr, dim=1).indices
    else:
        allowed = torch.arange(E)
        if w.empty_experts:
            empty = torch.randperm(E, generator=g)[: w.empty_experts]
            mask = torch.ones(E, dtype=torch.bool)
            mask[empty] = False
            allowed = allowed[mask]
        keys = torch.rand(T, len(allowed), generator=g)
        ids = allowed[torch.argsort(keys, dim=1)[:, :kr]]
    logits = torch.randn(T, kr, generator=g, dtype=torch.float32)
    p = torch.softmax(logits, dim=1)
    return ids.to(torch.int32).to(device), p.to(torch.float32).to(device)


def max_m_for(w: Workload, counts) -> int:
    """Masked slot capacity: the workload's max_m, raised to cover the largest expert
    (rounded up to 64) when the token count exceeds it (the host-weight sweep)."""
    mx = int(max(counts)) if len(counts) else 0
    return max(w.max_m, (mx + 63) // 64 * 64)
