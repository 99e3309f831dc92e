"""A C program (tests/c_abi_smoke.c), compiled by gcc against include/bsfroute.h and
linked with libbsfroute.so, runs the tiny workload end to end through the C ABI alone
(quantise weight -> prepare SF -> tile -> quantise -> route -> grouped GEMM -> combine
on cudaMalloc'd buffers).  Its output must match the oracle within the stated
tolerances and be bit-identical to the same path driven from Python."""

import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from block_scaled_fp8_route_gb300 import MoEPath, build
from tests.gpu_util import bits16, check_combined, require_gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _compile(out_path, syntax_only=False):
    cuda = _cuda_home()
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror", os.path.join(HERE, "c_abi_smoke.c"),
           "-I", os.path.join(build.ROOT, "include"), "-I", os.path.join(cuda, "include")]
    if syntax_only:
        cmd += ["-fsyntax-only"]
    else:
        lib_dir = os.path.dirname(build.LIB_PATH)
        cmd += ["-o", out_path, "-L", lib_dir, "-lbsfroute", "-Wl,-rpath," + lib_dir,
                "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr


def test_c_caller_compiles_against_the_header_alone():
    """No GPU needed: the header is valid C11 and declares everything the C caller uses."""
    _compile(None, syntax_only=True)


@pytest.mark.gpu
def test_c_caller_runs_the_path(tmp_path):
    dev = require_gpu()
    exe = str(tmp_path / "c_abi_smoke")
    _compile(exe)
    w = W.WORKLOADS["tiny_a128"]
    x, wt = W.activations(w), W.weights(w)
    ids, p = W.routing(w)
    bits16(x).tofile(tmp_path / "x.bin")
    bits16(wt).tofile(tmp_path / "w.bin")
    ids.numpy().astype(np.int32).tofile(tmp_path / "ids.bin")
    p.numpy().astype(np.float32).tofile(tmp_path / "p.bin")
    res = subprocess.run([exe, str(tmp_path), str(w.T), str(w.kr), str(w.E), str(w.K), str(w.N), str(w.align)],
                         capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    z_c = np.fromfile(tmp_path / "z.bin", dtype=np.uint16).reshape(w.T, w.N)
    oi_c = np.fromfile(tmp_path / "output_index.bin", dtype=np.int32).reshape(w.T, w.kr)

    # oracle
    aq, asf = oracle.quantise.quantise_act(bits16(x))
    bq, bsf = oracle.quantise.quantise_weight(bits16(wt))
    r = oracle.route.route(ids.numpy(), w.E, w.layout, align=w.align)
    assert np.array_equal(oi_c, r["output_index"])
    a_rows = oracle.route.scatter_rows(aq, r["token_of_row"])
    a_sf = oracle.route.scatter_rows(asf, r["token_of_row"], pad_value=127)
    y_ref, _ = oracle.gemm.grouped_gemm(a_rows, a_sf, bq, bsf, r["seg_start"], r["counts"])
    z_ref = oracle.combine.combine(y_ref, r["output_index"], p.numpy())
    rms = oracle.checks.expert_row_rms(oracle.formats.bf16_bits_to_f64(y_ref), r["seg_start"], r["counts"])
    check_combined(z_c, z_ref, y_ref, r["output_index"], p.numpy(), rms, "C caller combined output")

    # the same path from Python (same library, same kernels): bit-identical
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=w.align, device=dev,
                   fused_dispatch=False)
    z_py = path.step(x.to(dev), ids.to(dev), p.to(dev))
    torch.cuda.synchronize()
    assert np.array_equal(bits16(z_py), z_c)
