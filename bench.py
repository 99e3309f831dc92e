"""Benchmark of the MoE expert path on one GB300 (or N replicas, one per GPU).

One step = quantise_act -> route (+scatter) -> grouped GEMM(s) -> combine on
one batch of seeded synthetic inputs already resident in HBM.  Prints ONE JSON
line (rank 0).  Default workload: the masked decode batch (T=128, top-8 of
128 experts, K=4096, N=3072, max_m=64), metric HBM GB/s.  ``--workload
prefill|large`` times the large-M batches (metric TFLOPS).

--impl reference times the CPU oracle (float64 numpy restatement of the same
path) on a bounded sample of the same workload, on the host cores.
"""

import argparse
import collections
import contextlib
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "dram_traffic.json")
GEMM_SRC = os.path.join(ROOT, "block_scaled_fp8_route_gb300", "csrc", "gemm.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=["decode", "prefill", "large", "tiny", "host"])
    ap.add_argument("--tokens", default="16,32,64,128,256,512,1024,2048,4096",
                    help="token counts of the host-weight sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-formats", action="store_true",
                    help="skip the decode step in the other operand formats (default decode run)")
    ap.add_argument("--fmt", default="fp8", choices=["fp8", "nvfp4", "bf16", "fp8_f32sf"],
                    help="operand format: FP8 E4M3 with UE8M0 scales, NVFP4 (E2M1, UE4M3 per 16), BF16, "
                         "or FP8 with float32 scales")
    ap.add_argument("--no-fused-dispatch", action="store_true",
                    help="quantise + route as separate launches even where the single-launch dispatch applies")
    ap.add_argument("--no-route-quantise", action="store_true",
                    help="large FP8 batches: quantise + route with the token-major copy instead of the fused "
                         "route + quantise-scatter")
    ap.add_argument("--no-large-m", action="store_true",
                    help="skip the large-M GEMM measurements added to the decode line")
    ap.add_argument("--gemm", choices=["gate_up", "down"], default=None,
                    help="time one grouped GEMM of the workload (prefill / large) instead of the step; with "
                         "--experts, on the first n experts only (same rows per expert, K and N): the small "
                         "case of a profiler capture")
    ap.add_argument("--experts", type=int, default=0)
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


# ----------------------------------------------------------------------------- multi-rank helpers
def max_over_ranks(value, device="cpu"):
    """The largest value over all ranks (the slowest replica's time); identity on one rank."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_throughput(units_per_step, steps, world, elapsed_ms, scale):
    """Whole-job throughput: the units every replica processed over the slowest replica's time."""
    return units_per_step * steps * world / (elapsed_ms / 1e3) / scale


# ----------------------------------------------------------------------------- work accounting
DTYPES = {"fp8": "e4m3 x e4m3 -> f32 acc -> bf16",
          "nvfp4": "e2m1 x e2m1 (ue4m3 per 16, 2^j per tensor) -> f32 acc -> bf16",
          "bf16": "bf16 x bf16 -> f32 acc -> bf16",
          "fp8_f32sf": "e4m3 x e4m3 (f32 scales per 128-K block, applied on CUDA cores) -> f32 acc -> bf16"}


def operand_bytes(K, fmt):
    """(data bytes, scale bytes) of one quantised row of K values: FP8 K and one UE8M0 byte per
    128 packed four to a word; NVFP4 K/2 and one UE4M3 byte per 16."""
    if fmt == "nvfp4":
        return K // 2, K // 16
    if fmt == "bf16":
        return 2 * K, 0
    if fmt == "fp8_f32sf":
        return K, (K // 128) * 4
    return K, ((K // 128 + 3) // 4) * 4


def weight_bytes(N, K, fmt):
    """Bytes of one expert's weights and the weight scales the GEMM reads: per-row packed UE8M0
    words (FP8), per-row UE4M3 bytes (NVFP4), one float32 per 128 x 128 block (FP32 scales)."""
    if fmt == "fp8_f32sf":
        return N * K + (N // 128) * (K // 128) * 4
    qb, sb = operand_bytes(K, fmt)
    return N * (qb + sb)


def step_work(w, counts, placed_rows, fused_dispatch=False, fmt="fp8"):
    """Algorithmic bytes and GEMM flops of one step (valid rows only; padding excluded).
    With the single-launch dispatch or the fused route + quantise-scatter (stage "dispatch") the
    activations are read once and only the packed rows are written; otherwise the token-major
    quantised copy is written and re-read."""
    T, K, N, E, kr = w.T, w.K, w.N, w.E, w.kr
    R = T * kr
    qb, sb = operand_bytes(K, fmt)
    active = [int(c) for c in counts if c > 0]
    rows = sum(active)
    b = {}
    if fmt == "bf16":
        b["route"] = R * 4 + R * 4 + placed_rows * 8 + rows * 2 * qb       # indices + bf16 row copy
    elif fused_dispatch:
        b["dispatch"] = T * K * 2 + R * 4 + R * 4 + placed_rows * 8 + rows * (qb + sb)
    else:
        b["quantise"] = T * K * 2 + T * (qb + sb)
        b["route"] = R * 4 + R * 4 + placed_rows * 8 + rows * 2 * (qb + sb)
    gemm_bytes = len(active) * weight_bytes(N, K, fmt) + rows * (qb + sb + N * 2)
    flops = 2.0 * rows * N * K
    b["gemm"] = gemm_bytes
    out_n = N
    if w.K2:
        qb2, sb2 = operand_bytes(w.K2, fmt)
        if fmt == "fp8":   # only the routed rows of the packed input are quantised
            b["quantise2"] = rows * w.K2 * 2 + rows * (qb2 + sb2)
        elif fmt != "bf16":
            b["quantise2"] = placed_rows * w.K2 * 2 + placed_rows * (qb2 + sb2)
        b["gemm2"] = len(active) * weight_bytes(w.N2, w.K2, fmt) + rows * (qb2 + sb2 + w.N2 * 2)
        flops += 2.0 * rows * w.N2 * w.K2
        out_n = w.N2
    b["combine"] = R * out_n * 2 + T * out_n * 2 + R * 8
    return b, flops


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and throttle reasons sampled every ~0.2 ms through NVML (ctypes on the
    driver's libnvidia-ml) while the timed region runs (a few-millisecond region still
    gets tens of samples); nvidia-smi as a fallback."""

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None
        self.nvml = None
        self.handle = None
        self.max_mhz = None
        self.proc = None
        self.lines = []
        self.recording = threading.Event()   # samples are kept only between begin() and stop()

    def _init_nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(self.gpu).uuid)
        except Exception:
            uuid = None
        ok = False
        if uuid:
            u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            ok = lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(handle)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.gpu, ctypes.byref(handle)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))      # NVML_CLOCK_SM
        self.nvml, self.handle, self.max_mhz = lib, handle, float(mx.value)

    def _loop(self):
        import ctypes
        mhz = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        get_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_flag.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0:
                r = reasons.value if get_reasons(self.handle, ctypes.byref(reasons)) == 0 else 0
                if self.recording.is_set():
                    self.samples.append((float(mhz.value), int(r)))
            time.sleep(0.0002)

    def start(self):
        # the main thread mostly enqueues work while holding the GIL; a short switch interval lets
        # the sampling thread run every ~0.2 ms instead of every 5 ms (restored in stop())
        self.switch_interval = sys.getswitchinterval()
        sys.setswitchinterval(1e-4)
        try:
            self._init_nvml()
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
            return
        except (OSError, AttributeError):
            self.nvml = None
        try:
            fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                      "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                      "clocks_event_reasons.sw_power_cap")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={fields}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(
                target=lambda: [self.lines.append(x.strip()) for x in self.proc.stdout if self.recording.is_set()],
                daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def begin(self):
        """Start keeping samples (the thread started in start() is already running)."""
        self.recording.set()

    def stop(self):
        sys.setswitchinterval(getattr(self, "switch_interval", 0.005))
        if self.nvml is not None:
            self.stop_flag.set()
            self.thread.join(timeout=2)
            if not self.samples:
                return None
            reasons = set()
            for _, r in self.samples:
                for bit, name in self.REASONS.items():
                    if r & bit:
                        reasons.add(name)
            return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                    "reasons": sorted(reasons), "samples": len(self.samples), "source": "nvml"}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi"}


# ----------------------------------------------------------------------------- traffic record
def gemm_source_hash():
    h = hashlib.sha256()
    for name in ("gemm.cu", "common.cuh"):
        with open(os.path.join(ROOT, "block_scaled_fp8_route_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per GEMM launch from the committed ncu summary, if it matches this source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        rec = json.load(f)
    entry = rec.get(workload)
    if not entry or entry.get("gemm_source_hash") != gemm_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- oracle (CPU) leg
class OracleSample:
    """The CPU oracle on the path restricted to ``n_experts`` experts (the busiest ones).

    Inputs, including the oracle's quantisation of those experts' weights (a
    once-per-weight-load step), are prepared untimed; ``run()`` times one pass of
    quantise -> route -> scatter -> expert GEMMs -> combine and returns
    (seconds, algorithmic bytes, flops)."""

    def __init__(self, w, n_experts, fmt="fp8"):
        import oracle
        self.oracle = oracle
        self.w = w
        self.fmt = fmt
        x = W.activations(w)
        ids, p = W.routing(w)
        counts = np.bincount(ids.numpy().reshape(-1), minlength=w.E)
        self.experts = [int(e) for e in np.argsort(-counts, kind="stable")[:n_experts] if counts[e] > 0]
        wt = W.weights(w, experts=self.experts)
        self.xb = x.view(torch.int16).numpy().view(np.uint16)
        self.ids = ids.numpy()
        self.p = p.numpy()
        wb = wt.view(torch.int16).numpy().view(np.uint16)
        if fmt == "bf16":
            self.bq, self.bsf = wb, None
        elif fmt == "fp8_f32sf":
            self.bq, self.bsf = oracle.f32sf.quantise_weight(wb)
        elif fmt == "nvfp4":
            wv = oracle.formats.bf16_bits_to_f64(wb)
            self.bj = oracle.nvfp4.global_exponent(np.abs(wv).reshape(len(self.experts), -1).max(axis=1))
            self.bq, _, self.bsf = oracle.nvfp4.quantise_weight(wb, self.bj)
        else:
            self.bq, self.bsf = oracle.quantise.quantise_weight(wb)
        self.desc = (f"oracle (float64 numpy, {fmt}) over the {len(self.experts)} busiest of {w.E} experts; quantise, "
                     f"route, scatter and combine over the whole batch; first GEMM only")

    def run(self):
        o, w = self.oracle, self.w
        fp4, bf, f32 = self.fmt == "nvfp4", self.fmt == "bf16", self.fmt == "fp8_f32sf"
        t0 = time.perf_counter()
        if f32:
            aq, asf = o.f32sf.quantise_act(self.xb)
        elif bf:
            aq, asf = self.xb, np.zeros((self.xb.shape[0], 1), dtype=np.uint8)
        elif fp4:
            aq, _, asf = o.nvfp4.quantise_act(self.xb, 0)
        else:
            aq, asf = o.quantise.quantise_act(self.xb)
        r = o.route.route(self.ids, w.E, w.layout, align=w.align, max_m=w.max_m)
        a_rows = o.route.scatter_rows(aq, r["token_of_row"])
        a_sf = o.route.scatter_rows(asf, r["token_of_row"], pad_value=1.0 if f32 else 0 if fp4 else 127)
        y = np.zeros((r["rows_used"], w.N), dtype=np.uint16)
        rows = 0
        for i, e in enumerate(self.experts):
            s, c = int(r["seg_start"][e]), int(r["counts"][e])
            if f32:
                y[s:s + c], _ = o.f32sf.grouped_gemm(a_rows[s:s + c], a_sf[s:s + c], self.bq[i:i + 1],
                                                     self.bsf[i:i + 1], np.array([0, c]), np.array([c]))
            elif bf:
                y[s:s + c], _ = o.bf16.grouped_gemm(a_rows[s:s + c], self.bq[i:i + 1], np.array([0, c]),
                                                    np.array([c]))
            elif fp4:
                y[s:s + c], _ = o.nvfp4.grouped_gemm(a_rows[s:s + c], a_sf[s:s + c], 0, self.bq[i:i + 1],
                                                     self.bsf[i:i + 1], self.bj[i:i + 1], np.array([0, c]),
                                                     np.array([c]))
            else:
                y[s:s + c] = o.gemm.expert_gemm(a_rows[s:s + c], a_sf[s:s + c], self.bq[i], self.bsf[i])
            rows += c
        o.combine.combine(y, r["output_index"], self.p)
        dt = time.perf_counter() - t0
        qb, sb = operand_bytes(w.K, self.fmt)
        byts = len(self.experts) * weight_bytes(w.N, w.K, self.fmt) + rows * (qb + sb + w.N * 2)
        return dt, byts, 2.0 * rows * w.N * w.K


def workload_config(w, fmt="fp8"):
    """The ``config`` object of the JSON line (identical for both arms)."""
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    ids, _ = W.routing(w)
    counts = np.bincount(ids.numpy().reshape(-1), minlength=w.E)
    cfg = {"workload": w.name, "T": w.T, "top_k": w.kr, "experts": w.E, "K": w.K, "N": w.N,
           "layout": "masked" if w.layout == W.MASKED else "contiguous",
           "max_m" if w.layout == W.MASKED else "align": a_or_m,
           "l2": f"no flush: weights {(w.E * w.N * w.K) / 1e9:.2f} GB > 129 MB L2, streamed each step",
           "routed_rows": int(np.minimum(counts, a_or_m).sum()) if w.layout == W.MASKED else int(counts.sum()),
           "active_experts": int((counts > 0).sum())}
    if w.K2:
        cfg.update({"K2": w.K2, "N2": w.N2})
    if fmt != "fp8":
        cfg["format"] = fmt
        cfg["l2"] = f"no flush: weights {(w.E * weight_bytes(w.N, w.K, fmt)) / 1e9:.2f} GB > 129 MB L2, streamed each step"
    return cfg


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, w, metric, unit, hib):
    """--impl reference: the oracle as it stands, on the host cores."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    sample = OracleSample(w, 2 if w.name in ("decode", "host", "tiny") else 1, fmt=args.fmt)
    for _ in range(args.warmup):
        sample.run()
    tot_t, tot_b, tot_f = 0.0, 0.0, 0.0
    for _ in range(args.steps):
        dt, b, f = sample.run()
        tot_t += dt
        tot_b += b
        tot_f += f
    desc = sample.desc
    value = (tot_b / tot_t / 1e9) if unit == "GB/s" else (tot_f / tot_t / 1e12)
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": hib, "data": "synthetic", "dtype": "f64",
        "config": workload_config(w, args.fmt),
        "cpu_baseline": {"value": value, "unit": unit, "cores": host_cores(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- host-weight sweep
def measure_read_gbs(t, host_mapped, reps=5):
    """Bandwidth at which the SMs stream-read tensor t (device, or pinned host through its mapped address)."""
    from block_scaled_fp8_route_gb300 import ops
    out = torch.empty(1, dtype=torch.int64, device="cuda")
    for _ in range(2):
        ops.checksum_u64(t, host_mapped=host_mapped, out=out)
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        e0.record()
        ops.checksum_u64(t, host_mapped=host_mapped, out=out)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    return t.numel() * t.element_size() / (best / 1e3) / 1e9


def run_host_sweep(args, w, metric):
    """Grouped GEMM with every weight byte in pinned host memory, T swept; one JSON line."""
    from block_scaled_fp8_route_gb300 import MoEPath, ops, _lib
    _lib.load()
    dev = torch.device("cuda", 0)
    wt = W.weights(w, device=dev)
    probe = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()        # 1 GiB pinned probe buffer
    link_gbs = measure_read_gbs(probe, True)
    dprobe = torch.empty_like(probe, device=dev)
    dprobe.copy_(probe, non_blocking=True)          # first copy maps the destination: untimed
    torch.cuda.synchronize()
    best_ms = None
    for _ in range(3):
        h2d_t0, h2d_t1 = torch.cuda.Event(True), torch.cuda.Event(True)
        h2d_t0.record()
        dprobe.copy_(probe, non_blocking=True)
        h2d_t1.record()
        torch.cuda.synchronize()
        ms = h2d_t0.elapsed_time(h2d_t1)
        best_ms = ms if best_ms is None else min(best_ms, ms)
    memcpy_gbs = probe.numel() / (best_ms / 1e3) / 1e9
    del dprobe
    sweep = []
    path = None
    wq_h = sfb_h = None
    clocks = ClockSampler(0)
    clocks.start()
    clocks.begin()
    for T in [int(v) for v in args.tokens.split(",")]:
        wT = W.with_tokens(w, T)
        ids, p = W.routing(wT, device=dev)
        counts = torch.bincount(ids.flatten().long(), minlength=w.E).cpu().numpy()
        max_m = W.max_m_for(wT, counts)
        x = W.activations(wT, device=dev)
        path = MoEPath(w.E, w.kr, T, w.K, w.N, wt if wq_h is None else wt[:1], layout=W.MASKED,
                       align_or_max_m=max_m, device=dev, weights_on_host=True, expected_m=T * w.kr // w.E)
        if wq_h is None:
            wq_h, sfb_h = path.wq, path.sfb
        else:
            path.wq, path.sfb = wq_h, sfb_h
        for _ in range(args.warmup):
            path.step(x, ids, p)
        torch.cuda.synchronize()
        ev = []
        orig = path.gemm

        def timed(*a, **k):
            e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
            e0.record()
            r = orig(*a, **k)
            e1.record()
            ev.append((e0, e1))
            return r

        path.gemm = timed
        s0, s1 = torch.cuda.Event(True), torch.cuda.Event(True)
        s0.record()
        for _ in range(args.steps):
            path.step(x, ids, p)
        s1.record()
        torch.cuda.synchronize()
        path.gemm = orig
        assert ops.device_error() == 0
        gemm_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        active = int((counts > 0).sum())
        nw = (w.K // 128 + 3) // 4
        link_bytes = active * (w.N * w.K + w.N * nw * 4)
        rows = int(np.minimum(counts, max_m).sum())
        flops = 2.0 * rows * w.N * w.K
        sweep.append({"T": T, "max_m": max_m, "active_experts": active, "gemm_ms": gemm_ms,
                      "step_ms": s0.elapsed_time(s1) / args.steps,
                      "link_gbs": link_bytes / (gemm_ms / 1e3) / 1e9, "tflops": flops / (gemm_ms / 1e3) / 1e12})
    clk = clocks.stop()
    last = sweep[-1]
    # end to end at the last T: pinned host batches in, output back, every step (HostStreamedPath)
    from block_scaled_fp8_route_gb300 import HostStreamedPath
    wl = W.with_tokens(w, last["T"])
    x_h = W.activations(wl).pin_memory()
    ids_h, p_h = (t.pin_memory() for t in W.routing(wl))
    streamed = HostStreamedPath(path, wl.T, wl.K, wl.kr, device=dev)
    outs = [torch.empty(path.z.shape, dtype=path.z.dtype).pin_memory() for _ in range(4)]
    batches = [(x_h, ids_h, p_h)] * args.steps
    streamed.run(batches[:2], outs[:2])
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(True), torch.cuda.Event(True)
    streamed.run(batches, [outs[i % 4] for i in range(args.steps)], start_event=s0, end_event=s1)
    torch.cuda.synchronize()
    e2e_ms = s0.elapsed_time(s1) / args.steps
    link_bytes_last = last["link_gbs"] * last["gemm_ms"] / 1e3 * 1e9
    e2e = {"value": link_bytes_last / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (x_h, ids_h, p_h)),
           "d2h_bytes_per_step": outs[0].numel() * outs[0].element_size(), "ms_per_step": e2e_ms,
           "how": "pinned host batches -> device -> whole path (graph, weights read from host memory) -> "
                  "pinned host output, every step (HostStreamedPath)"}
    del streamed
    # the oracle on a bounded sample of the same T (the busiest two experts), on the host cores
    cpu = None
    if not args.no_cpu_baseline:
        sample = OracleSample(wl, 2)
        tot_t = tot_b = 0.0
        reps = 0
        while tot_t < 10.0 and reps < 50:
            dt, b, _ = sample.run()
            tot_t, tot_b, reps = tot_t + dt, tot_b + b, reps + 1
        cpu = {"value": tot_b / tot_t / 1e9, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"{sample.desc}; T={wl.T}; {reps} passes; bytes = weights and rows of the sampled experts",
               "seconds": tot_t}
    line = {
        "metric": metric, "value": last["link_gbs"], "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": last["step_ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32 acc -> bf16", "data": "synthetic",
        "config": {"workload": "host", "T": last["T"], "top_k": w.kr, "experts": w.E, "K": w.K, "N": w.N,
                   "layout": "masked", "weights": "pinned host memory, read in-kernel through mapped addresses"},
        "roofline": {"bound": "host-link", "achieved": last["link_gbs"], "peak": link_gbs, "unit": "GB/s",
                     "frac": last["link_gbs"] / link_gbs, "peak_src": "measured SM stream read of 1 GiB pinned host memory",
                     "traffic": None, "kernel": "grouped_gemm_kernel"},
        "host_link": {"sm_read_gbs": link_gbs, "memcpy_h2d_gbs": memcpy_gbs},
        "sweep": sweep, "clocks": clk, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": path.launches_per_step() * args.steps,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- large-M GEMMs (context object)
def tensor_peak_tflops(pk, fmt):
    """Dense tensor peak of a format: the measured bf16 burst times the nominal ratio of the
    format's rate to bf16 (FP8 and FP8 with float32 scales 2x, NVFP4 6x: 4.5 / 13.5 vs 2.25 PF)."""
    return pk["bf16_tflops"] * {"fp8": 2.0, "fp8_f32sf": 2.0, "nvfp4": 6.0, "bf16": 1.0}[fmt]


def _format_operands(fmt, x, wt, K):
    """Quantised (or bf16) activations and tiled weights of one format, and a GEMM closure."""
    from block_scaled_fp8_route_gb300 import ops
    if fmt == "bf16":
        bq = ops.tile_weights(wt.contiguous())
        return lambda seg, cnt, d: ops.grouped_gemm_bf16_contig(x, bq, seg, cnt, d=d, flags=ops.B_TILED)
    if fmt == "nvfp4":
        aq, asf = ops.quantise_act_nvfp4(x, 0)
        bq, sfb, b_exp = ops.quantise_weight_nvfp4(wt)
        bq = ops.tile_weights(bq)
        return lambda seg, cnt, d: ops.grouped_gemm_nvfp4_contig(aq, asf, 0, bq, sfb, b_exp, seg, cnt, d=d,
                                                                 flags=ops.B_TILED)
    if fmt == "fp8_f32sf":
        aq, asf = ops.quantise_act_f32sf(x)
        bq, sfb = ops.quantise_weight_f32sf(wt)
        bq = ops.tile_weights(bq)
        return lambda seg, cnt, d: ops.grouped_gemm_f32sf_contig(aq, asf, bq, sfb, seg, cnt, d=d, flags=ops.B_TILED)
    aq, asf = ops.quantise_act(x)
    bq, sf128 = ops.quantise_weight(wt)
    bq = ops.tile_weights(bq)
    sfb = ops.prepare_weight_sf(sf128, K)
    return lambda seg, cnt, d: ops.grouped_gemm_contig(aq, asf, bq, sfb, seg, cnt, d=d, flags=ops.B_TILED)


def large_m_gemms(dev, pk, reps=10, fmts=("fp8",)):
    """Gate-up and down grouped GEMMs of the prefill and large workloads, timed alone (CUDA events
    on the launch stream), in each operand format against its own tensor peak and byte roofline,
    plus a library FP8 GEMM for context."""
    from block_scaled_fp8_route_gb300 import ops
    out = {}
    for fmt in fmts:
        peak = tensor_peak_tflops(pk, fmt)
        res_f = {}
        for name in ("prefill", "large"):
            w = W.WORKLOADS[name]
            ids, _ = W.routing(w, device=dev)
            bufs = ops.route(ids, w.E, w.layout, w.align)
            rows = int(bufs.counts.sum().item())
            active = int((bufs.counts > 0).sum().item())
            res = {}
            for tag, (K, N) in enumerate(((w.K, w.N), (w.K2, w.N2))):
                x = W.activations(W.with_tokens(w, bufs.m_cap), device=dev, K=K, tag=tag)
                wt = W.weights(w, device=dev, N=N, K=K, tag=tag)
                gemm = _format_operands(fmt, x, wt, K)
                del x, wt
                torch.cuda.empty_cache()
                d = torch.empty((bufs.m_cap, N), dtype=torch.bfloat16, device=dev)
                for _ in range(3):
                    gemm(bufs.seg_start, bufs.counts, d)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
                e0.record()
                for _ in range(reps):
                    gemm(bufs.seg_start, bufs.counts, d)
                e1.record()
                torch.cuda.synchronize()
                assert ops.device_error() == 0
                ms = e0.elapsed_time(e1) / reps
                tf = 2.0 * rows * N * K / (ms / 1e3) / 1e12
                qb, sb = operand_bytes(K, fmt)
                nbytes = active * weight_bytes(N, K, fmt) + rows * (qb + sb + 2 * N)
                rf = binding_roofline(2.0 * rows * N * K, nbytes, ms, peak, pk["hbm_gbs"])
                res["gate_up" if tag == 0 else "down"] = {"K": K, "N": N, "ms": ms, "tflops": tf, "frac": tf / peak,
                                                          "bytes": nbytes, "bound": rf["bound"],
                                                          "roofline_frac": rf["roofline_frac"]}
                del gemm, d
                torch.cuda.empty_cache()
            res_f[name] = {"routed_rows": rows, **res}
        res_f["tensor_peak_tflops"] = peak
        res_f["tensor_peak_src"] = f"{tensor_peak_tflops(pk, fmt) / pk['bf16_tflops']:g} x bf16 burst ({pk['src']})"
        out[fmt] = res_f
    if "fp8" in out:   # the FP8 entry keeps its historical flat layout
        f = out.pop("fp8")
        out.update({"prefill": f["prefill"], "large": f["large"], "fp8_peak_tflops": f["tensor_peak_tflops"],
                    "fp8_peak_src": f["tensor_peak_src"]})
    try:   # library FP8 GEMM (cuBLASLt through torch) for context only
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b.t(), one, one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
            e0.record()
            torch._scaled_mm(a, b.t(), one, one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        out["library_fp8_8192_tflops"] = 2.0 * n ** 3 / (best / 1e3) / 1e12
    except Exception as exc:   # pragma: no cover - depends on the torch build
        out["library_fp8_8192_tflops"] = None
        out["library_fp8_note"] = str(exc)[:120]
    return out


def binding_roofline(flops, nbytes, ms, tensor_peak_tflops, hbm_peak_gbs):
    """The roofline a launch sits under: t_F = flops / tensor peak against t_B = bytes / HBM
    bandwidth; the larger one binds.  Returns the roofline object in the binding unit plus the
    fraction of the tensor peak and max(t_F, t_B) / t (the "% of roofline")."""
    t = ms / 1e3
    t_f = flops / (tensor_peak_tflops * 1e12)
    t_b = nbytes / (hbm_peak_gbs * 1e9)
    if t_b > t_f:
        roof = {"bound": "hbm", "achieved": nbytes / t / 1e9, "peak": hbm_peak_gbs, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / t / 1e12, "peak": tensor_peak_tflops, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["tensor_frac"] = flops / t / 1e12 / tensor_peak_tflops
    roof["roofline_frac"] = max(t_f, t_b) / t
    return roof


def decode_formats(dev, pk, steps=50):
    """The decode step in the other operand formats (NVFP4, BF16, FP8 with float32 scales): the
    grouped GEMM timed alone over eager steps (CUDA events around its launch) and the whole step as
    CUDA-graph replays, bytes from each format's own accounting."""
    from block_scaled_fp8_route_gb300 import MoEPath
    w = W.WORKLOADS["decode"]
    ids, p = W.routing(w, device=dev)
    x = W.activations(w, device=dev)
    out = {}
    for fmt in ("nvfp4", "bf16", "fp8_f32sf"):
        wt = W.weights(w, device=dev)
        path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=w.max_m, device=dev,
                       expected_m=w.T * w.kr // w.E, fmt=fmt)
        del wt
        torch.cuda.empty_cache()
        path.step(x, ids, p)
        torch.cuda.synchronize()
        counts = path.bufs.counts.cpu().numpy()
        placed = int(path.bufs.seg_start[-1].item())
        byts, _ = step_work(w, counts, placed, fused_dispatch=path.fused_dispatch or path.route_quantise, fmt=fmt)
        ev = []
        orig = path.gemm

        def timed(*a, **k):
            e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
            e0.record()
            r = orig(*a, **k)
            e1.record()
            ev.append((e0, e1))
            return r

        path.gemm = timed
        for _ in range(steps):
            path.step(x, ids, p)
        torch.cuda.synchronize()
        path.gemm = orig
        gemm_ms = statistics.mean(a.elapsed_time(b) for a, b in ev[3:])
        path.capture(x, ids, p)
        for _ in range(3):
            path.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        e0.record()
        for _ in range(steps):
            path.replay()
        e1.record()
        torch.cuda.synchronize()
        step_ms = e0.elapsed_time(e1) / steps
        from block_scaled_fp8_route_gb300 import ops
        assert ops.device_error() == 0
        gbs = byts["gemm"] / (gemm_ms / 1e3) / 1e9
        out[fmt] = {"gemm_ms": gemm_ms, "gemm_gbs": gbs, "gemm_frac": gbs / pk["hbm_gbs"],
                    "gemm_bytes": byts["gemm"], "step_ms": step_ms,
                    "step_gbs": sum(byts.values()) / (step_ms / 1e3) / 1e9, "dtype": DTYPES[fmt]}
        del path
        torch.cuda.empty_cache()
    out["peak_gbs"] = pk["hbm_gbs"]
    return out


# ----------------------------------------------------------------------------- GPU leg
def run_gemm_case(args, w):
    """One grouped GEMM of a prefill / large workload (operand format --fmt, tiled weights, the step's
    launch configuration), optionally on its first n experts: --warmup untimed launches, then --steps timed
    ones (CUDA events); prints one JSON line with the time and the binding roofline."""
    from block_scaled_fp8_route_gb300 import ops, _lib
    _lib.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk = peaks()
    ids, _ = W.routing(w, device=dev)
    full = ops.route(ids, w.E, w.layout, w.align)
    ne = args.experts if args.experts > 0 else w.E
    counts = full.counts[:ne].clone()
    seg = torch.zeros(ne + 1, dtype=torch.int32, device=dev)
    seg[1:] = torch.cumsum((counts + w.align - 1) // w.align * w.align, 0)
    m = int(seg[-1].item())
    tag = 0 if args.gemm == "gate_up" else 1
    K, N = (w.K, w.N) if tag == 0 else (w.K2, w.N2)
    x = W.activations(W.with_tokens(w, m), device=dev, K=K, tag=tag)
    wt = W.weights(W.Workload(**{**w.__dict__, "E": ne}), device=dev, N=N, K=K, tag=tag)   # experts 0 .. ne-1
    gemm = _format_operands(args.fmt, x, wt, K)
    del x, wt
    torch.cuda.empty_cache()
    d = torch.empty((m, N), dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup):
        gemm(seg, counts, d)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
    e0.record()
    for _ in range(args.steps):
        gemm(seg, counts, d)
    e1.record()
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    ms = e0.elapsed_time(e1) / args.steps
    rows = int(counts.sum().item())
    active = int((counts > 0).sum().item())
    qb, sb = operand_bytes(K, args.fmt)
    nbytes = active * weight_bytes(N, K, args.fmt) + rows * (qb + sb + 2 * N)
    flops = 2.0 * rows * N * K
    roof = binding_roofline(flops, nbytes, ms, tensor_peak_tflops(pk, args.fmt), pk["hbm_gbs"])
    print(json.dumps({"workload": w.name, "gemm": args.gemm, "fmt": args.fmt, "experts": ne, "active_experts": active,
                      "routed_rows": rows, "K": K, "N": N, "ms": ms, "tflops": flops / (ms / 1e3) / 1e12,
                      "algorithmic_bytes": nbytes, "roofline": roof}), flush=True)


def main():
    args = parse()
    w = W.WORKLOADS[args.workload]
    if args.gemm is not None and args.impl != "reference":
        assert w.name in ("prefill", "large"), "--gemm applies to the prefill and large workloads"
        run_gemm_case(args, w)
        return
    if args.workload == "host" and args.impl != "reference":
        run_host_sweep(args, w, "grouped-GEMM TFLOPS & % FP8 roofline (large M); HBM GB/s & % peak (decode)")
        return
    large_m = w.name in ("prefill", "large")
    metric = "grouped-GEMM TFLOPS & % FP8 roofline (large M); HBM GB/s & % peak (decode)"
    unit = "TFLOP/s" if large_m else "GB/s"
    if args.impl == "reference":
        run_reference(args, w, metric, unit, True)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from block_scaled_fp8_route_gb300 import MoEPath, ops, _lib
    _lib.load()      # fails loudly if the CUDA library was not built

    pk = peaks()
    ids, p = W.routing(w, device=dev)
    x = W.activations(w, device=dev)
    wt = W.weights(w, device=dev)
    wt2 = W.weights(w, device=dev, N=w.N2, K=w.K2, tag=1) if w.K2 else None
    a_or_m = w.max_m if w.layout == W.MASKED else w.align
    expected_m = w.T * w.kr // w.E
    path = MoEPath(w.E, w.kr, w.T, w.K, w.N, wt, layout=w.layout, align_or_max_m=a_or_m, w2_bf16=wt2,
                   device=dev, expected_m=expected_m, fused_dispatch=False if args.no_fused_dispatch else None,
                   fmt=args.fmt, route_quantise=False if args.no_route_quantise else None)
    del wt, wt2
    torch.cuda.empty_cache()
    h2 = W.activations(W.with_tokens(w, path.bufs.m_cap), device=dev, K=w.K2, tag=1) if w.K2 else None
    stream = torch.cuda.current_stream()

    # routing counts for the work accounting (untimed)
    path.step(x, ids, p, h2)
    torch.cuda.synchronize()
    counts = path.bufs.counts.cpu().numpy()
    placed = int(path.bufs.seg_start[-1].item())
    assert ops.device_error() == 0, "device error during setup"
    bytes_by_kernel, flops = step_work(w, counts, placed, fused_dispatch=path.fused_dispatch or path.route_quantise,
                                       fmt=args.fmt)
    step_bytes = sum(bytes_by_kernel.values())

    for _ in range(args.warmup):
        path.step(x, ids, p, h2)

    # eager steps, with CUDA events around every stage (dispatch / quantise / route, GEMMs, combine)
    # on the launching stream
    stage_events = collections.defaultdict(list)

    @contextlib.contextmanager
    def stage_timer(name):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        yield
        e1.record(stream)
        stage_events[name].append((e0, e1))

    torch.cuda.synchronize()
    q0 = torch.cuda.Event(enable_timing=True)
    q1 = torch.cuda.Event(enable_timing=True)
    q0.record(stream)
    for _ in range(args.steps):
        path.step(x, ids, p, h2, timer=stage_timer)
    q1.record(stream)
    torch.cuda.synchronize()
    eager_ms = q0.elapsed_time(q1) / args.steps

    # the timed region: the same step replayed from a CUDA graph (launch gaps removed)
    path.capture(x, ids, p, h2)
    clocks = ClockSampler(local)
    clocks.start()                       # the sampling thread warms up during the warm-up replays
    for _ in range(args.warmup):
        path.replay()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.begin()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        path.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), dev)
    assert ops.device_error() == 0, "device error during the timed steps"

    stage_ms = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in stage_events.items()}
    # dominant kernel: the first (gate-up) GEMM
    first_gemm_ms = stage_ms["gemm"]
    per_kernel = {k: {"bytes": bytes_by_kernel[k], "us": stage_ms[k] * 1e3,
                      "gbs": bytes_by_kernel[k] / (stage_ms[k] / 1e3) / 1e9}
                  for k in stage_ms if k in bytes_by_kernel}
    launches_per_step = path.launches_per_step()

    if large_m:
        value = job_throughput(flops, args.steps, world, elapsed_ms, 1e12)
        # dense peak of the operand type: the measured bf16 burst x the nominal ratio (fp8 4.5 / 2.25 = 2,
        # fp4 13.5 / 2.25 = 6)
        ratio = {"nvfp4": 6.0, "fp8": 2.0, "fp8_f32sf": 2.0, "bf16": 1.0}[args.fmt]
        fp8_peak = ratio * pk["bf16_tflops"]
        gflops = 2.0 * int(counts.sum()) * w.N * w.K
        # near the ridge point: the gate-up GEMM's binding roofline (flops / tensor peak against
        # algorithmic bytes / HBM bandwidth)
        roof = binding_roofline(gflops, bytes_by_kernel["gemm"], first_gemm_ms, fp8_peak, pk["hbm_gbs"])
        roof["peak_src"] = (f"{ratio:g} x bf16 burst ({pk['src']})" if roof["bound"] == "tensor"
                            else pk["src"]) + f"; tensor peak {fp8_peak:.0f} TFLOP/s = {ratio:g} x bf16 burst"
    else:
        value = job_throughput(step_bytes, args.steps, world, elapsed_ms, 1e9)
        achieved = bytes_by_kernel["gemm"] / (first_gemm_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_src": pk["src"]}
    roof["traffic"] = recorded_traffic(w.name if args.fmt == "fp8" else f"{w.name}_{args.fmt}")
    roof["kernel"] = "grouped_gemm_kernel"
    roof["algorithmic_per_launch"] = bytes_by_kernel["gemm"] if not large_m else 2.0 * int(counts.sum()) * w.N * w.K
    roof["launch_ms"] = first_gemm_ms

    # ---------------------------------------------------------------- end to end through the public API
    # Every step copies its inputs from pinned host memory and reads its output back; the copies of
    # neighbouring steps overlap the current step's kernels (HostStreamedPath: two buffer sets, one
    # graph per set, a copy stream).
    e2e = None
    if not args.no_e2e:
        from block_scaled_fp8_route_gb300 import HostStreamedPath
        streamed = HostStreamedPath(path, w.T, w.K, w.kr, h2=h2, device=dev)
        nb = 4                       # separate pinned host buffers (same batch contents: exact byte accounting)
        batches = [(x.cpu().pin_memory(), ids.cpu().pin_memory(), p.cpu().pin_memory()) for _ in range(nb)]
        outs = [torch.empty(path.z.shape, dtype=path.z.dtype).pin_memory() for _ in range(nb)]
        h2d = sum(t.numel() * t.element_size() for t in batches[0])
        d2h = outs[0].numel() * outs[0].element_size()
        seq_in = [batches[i % nb] for i in range(args.steps)]
        seq_out = [outs[i % nb] for i in range(args.steps)]
        streamed.run(seq_in[: args.warmup] or seq_in[:1], seq_out[: args.warmup] or seq_out[:1])
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        streamed.run(seq_in, seq_out, start_event=s0, end_event=s1)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(s0.elapsed_time(s1), dev)
        ev = job_throughput(flops, args.steps, world, e_ms, 1e12) if large_m else \
            job_throughput(step_bytes, args.steps, world, e_ms, 1e9)
        e2e = {"value": ev, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / args.steps,
               "how": "pinned host batches -> device -> whole path (graph) -> pinned host output, every step; "
                      "copies of neighbouring steps overlap the current step (HostStreamedPath)"}
        del streamed

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = OracleSample(w, 16 if w.name == "decode" else 3, fmt=args.fmt)
        tot_t = tot_b = tot_f = 0.0
        reps = 0
        while tot_t < 10.0 and reps < 50:          # about 10 s of oracle time
            dt, b, f = sample.run()
            tot_t, tot_b, tot_f, reps = tot_t + dt, tot_b + b, tot_f + f, reps + 1
        cv = (tot_f / tot_t / 1e12) if large_m else (tot_b / tot_t / 1e9)
        cpu = {"value": cv, "unit": unit, "cores": host_cores(), "kind": "oracle",
               "sample": f"{sample.desc}; {reps} passes", "seconds": tot_t}

    # context: the rate at which the SMs stream-read HBM alone (this library's checksum kernel over
    # 4 GiB); the roofline's denominator stays the measured copy bandwidth
    hbm_read = None
    if rank == 0 and not large_m:
        probe = torch.empty(4 << 30, dtype=torch.uint8, device=dev)
        probe.fill_(1)
        hbm_read = measure_read_gbs(probe, False)
        del probe
        torch.cuda.empty_cache()

    formats = None
    if rank == 0 and world == 1 and w.name == "decode" and args.fmt == "fp8" and not args.no_formats:
        del path
        torch.cuda.empty_cache()
        path = None
        formats = decode_formats(dev, pk)

    large_m = None
    if rank == 0 and world == 1 and w.name == "decode" and args.fmt == "fp8" and not args.no_large_m:
        del path
        torch.cuda.empty_cache()
        large_m = large_m_gemms(dev, pk, fmts=("fp8", "nvfp4", "bf16", "fp8_f32sf"))
    if rank == 0:
        cfg = workload_config(w, args.fmt)
        line = {
            "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPES[args.fmt],
            "data": "synthetic", "config": cfg,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": launches_per_step * args.steps,
            "step_bytes": step_bytes, "step_gemm_flops": flops, "eager_ms_per_step": eager_ms,
            "timed": "CUDA-graph replays of the whole step (eager step time in eager_ms_per_step)",
            "large_m_gemm": large_m if large_m is not None else None,
            "per_kernel": per_kernel,
            "hbm_stream_read_gbs": hbm_read,
            "decode_formats": formats,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
