"""CPU oracle for the FP8 block-scaled MoE routing + grouped GEMM path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, deliberately
unoptimised restatement of what the hot path computes, written in numpy with
float64 arithmetic.  It exists to check the CUDA path, never to stand in for
it: only the test suite, the smoke check in ``__graft_entry__`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import it.  It shares no
code with the CUDA library and imports nothing from it.

Sources (page title, section):

* "GEMM 执行方式" (rainlin-net), §4.1 grouped GEMM as P independent problems,
  §4.2 top-k routing tensors, §4.3 packed layout, §4.4 expert GEMM and combine,
  §4.6 the 128-row aligned layout, scatter and gather.
* "FP8 的「不可能三角」被打破了" (DeepGEMM article, nxmr.cn), sections
  "FP8 的精度陷阱" (E4M3 format), "补偿机制一" (power-of-two scale factors,
  UE8M0 packing), "补偿机制三" (MN-major packed SF layout), "精度与吞吐的平衡点"
  (calc_diff tolerance, repeat-run determinism).
* "AsymGEMM" README, "Token Layout Protocols" (contiguous and masked layouts),
  "FP4 Asymmetric GEMM" (NVFP4 operands, ``oracle/nvfp4.py``), "BF16 Asymmetric
  GEMM" (``oracle/bf16.py``), notation ``disable_ue8m0_cast`` (float32 scale
  factors, ``oracle/f32sf.py``).
* "CuTeDSL bei Perplexity", Blackwell support (16-element absolute maximum
  of the NVFP4 quantiser).

Pinning status of each function is stated in its module docstring.  Every
function is pinned by at least one test in ``tests/test_oracle_*.py`` against
values the pages print, closed forms, library routines or brute force, except
the GPU-internal FP32 accumulation order, which is outside the oracle.
"""

from . import formats, quantise, route, gemm, combine, checks, nvfp4, bf16, f32sf  # noqa: F401
