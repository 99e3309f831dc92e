"""One pass of the MoE expert path on resident buffers.

    x bf16 [T, K] --quantise_act--> (q, sf) --route(+scatter)--> packed A
      --grouped GEMM (contiguous or masked)--> y bf16 --combine--> z bf16 [T, N]

with an optional second grouped GEMM (the down projection, K2 x N2) on a
separately supplied packed bf16 input that shares the routing; then the
combine reads the second GEMM's output.  Weights are quantised once at
construction (``quantise_weight`` + ``prepare_weight_sf``, or
``quantise_weight_nvfp4`` with ``fmt="nvfp4"``).  Every step is a
``libbsfroute.so`` call; this class only owns buffers and orders the calls on
one stream.
"""

import contextlib

import torch

from . import ops


@contextlib.contextmanager
def _no_timer(name):
    yield


class MoEPath:
    """``fmt`` = "fp8" (E4M3, UE8M0 per 1 x 128 / 128 x 128), "nvfp4" (E2M1, UE4M3 per 1 x 16, a
    power-of-two tensor exponent per expert for the weights and ``a_exp`` for the activations) or
    "bf16" (unquantised operands; the route scatters bf16 rows) or "fp8_f32sf" (E4M3 with float32
    scales, applied per 128-K block in software)."""

    def __init__(self, E, kr, T, K, N, w_bf16, layout=ops.CONTIGUOUS, align_or_max_m=1, w2_bf16=None,
                 device="cuda", weights_on_host=False, expected_m=0, fused_dispatch=None, fmt="fp8", a_exp=0,
                 tiled_weights=True, route_quantise=None):
        self.E, self.kr, self.T, self.K, self.N = E, kr, T, K, N
        self.layout, self.align_or_max_m = layout, align_or_max_m
        self.expected_m = expected_m
        self.fmt, self.a_exp = fmt, a_exp
        self.flags = (ops.B_HOST_MAPPED if weights_on_host else 0) | (ops.B_TILED if tiled_weights else 0)
        self.wq, self.sfb, self.b_exp = self._weights(w_bf16.to(device), K)
        if weights_on_host:
            self.wq = self.wq.cpu().pin_memory()
            self.sfb = self.sfb.cpu().pin_memory()
        self.two_gemms = w2_bf16 is not None
        if self.two_gemms:
            _, self.N2, self.K2 = w2_bf16.shape
            self.w2q, self.sfb2, self.b2_exp = self._weights(w2_bf16.to(device), self.K2)
        self.bufs = ops.RouteBuffers(T, kr, E, layout, align_or_max_m, K=K, device=device, fmt=fmt)
        self.fused_dispatch = ops.dispatch_supported(T, kr, E) if fused_dispatch is None else fused_dispatch
        if fmt in ("bf16", "fp8_f32sf"):
            self.fused_dispatch = False          # the route scatters the rows (bf16, or e4m3 + float32 scales)
        # FP8 batches above the single-launch limit: route, then quantise each token once into its k_r
        # packed rows (bsf_route_quantise) instead of quantise + route with a token-major copy
        auto_rq = fmt == "fp8" and not self.fused_dispatch and ops.route_quantise_supported(kr)
        self.route_quantise = auto_rq if route_quantise is None else (route_quantise and auto_rq)
        m = self.bufs.m_cap
        self.q, self.sf = self._act_buffers(T, K, device)
        self.y = torch.empty((max(m, 1), N), dtype=torch.bfloat16, device=device)
        if self.two_gemms:
            self.q2, self.sf2 = self._act_buffers(max(m, 1), self.K2, device)
            self.y2 = torch.empty((max(m, 1), self.N2), dtype=torch.bfloat16, device=device)
            self.z = torch.empty((T, self.N2), dtype=torch.bfloat16, device=device)
        else:
            self.z = torch.empty((T, N), dtype=torch.bfloat16, device=device)

    def _weights(self, w, K):
        wq, sfb, b_exp = self._quantised_weights(w, K)
        if self.flags & ops.B_TILED:
            wq = ops.tile_weights(wq)
        return wq, sfb, b_exp

    def _quantised_weights(self, w, K):
        if self.fmt == "bf16":
            return w.contiguous(), None, None
        if self.fmt == "fp8_f32sf":
            wq, sf = ops.quantise_weight_f32sf(w)
            return wq, sf, None
        if self.fmt == "nvfp4":
            return ops.quantise_weight_nvfp4(w)
        wq, sf128 = ops.quantise_weight(w)
        return wq, ops.prepare_weight_sf(sf128, K), None

    def _act_buffers(self, rows, K, device):
        if self.fmt == "bf16":
            return None, None
        if self.fmt == "fp8_f32sf":
            return (torch.empty((rows, K), dtype=torch.uint8, device=device),
                    torch.empty((K // 128, ops.sf_ld(rows)), dtype=torch.float32, device=device))
        if self.fmt == "nvfp4":
            return (torch.empty((rows, K // 2), dtype=torch.uint8, device=device),
                    torch.empty((K // 64, ops.sf_ld(rows)), dtype=torch.int32, device=device))
        return (torch.empty((rows, K), dtype=torch.uint8, device=device),
                torch.empty((ops.sf_words(K), ops.sf_ld(rows)), dtype=torch.int32, device=device))

    def _quantise(self, x, q, sf, rows=None):
        if self.fmt == "fp8_f32sf":
            return ops.quantise_act_f32sf(x, q=q, sf=sf)
        if self.fmt == "nvfp4":
            return ops.quantise_act_nvfp4(x, self.a_exp, q=q, sf=sf)
        return ops.quantise_act(x, q=q, sf=sf, rows=rows)

    def launches_per_step(self):
        """Kernel launches one ``step`` makes (all of them this library's kernels)."""
        R = self.T * self.kr
        if ops.dispatch_supported(self.T, self.kr, self.E):
            route = 2                                              # route_small + fill
        else:
            route = 3 + (1 if (R + 2047) // 2048 > 64 else 0)      # count + assign + fill (+ scan)
        if self.fused_dispatch:
            n = 1                                                  # dispatch
        elif self.route_quantise:
            # (up to 64 chunks the assign kernel marks the padding rows itself: no fill launch)
            small = ops.dispatch_supported(self.T, self.kr, self.E)
            n = route + 1 - (0 if small or (R + 2047) // 2048 > 64 else 1)   # routing + quantise-scatter
        else:
            n = (0 if self.fmt == "bf16" else 1) + route           # quantise + routing
        n += 1                                                     # grouped GEMM
        if self.two_gemms:
            n += 1 if self.fmt == "bf16" else 2                    # (quantise of h2 +) second GEMM
        return n + 1                                               # combine

    def gemm(self, a, sfa, wq, sfb, d, b_exp=None):
        b = self.bufs
        if self.fmt == "bf16":
            if self.layout == ops.MASKED:
                return ops.grouped_gemm_bf16_masked(a, wq, b.counts, self.align_or_max_m, d=d,
                                                    expected_m=self.expected_m, flags=self.flags)
            return ops.grouped_gemm_bf16_contig(a, wq, b.seg_start, b.counts, d=d, flags=self.flags)
        if self.fmt == "fp8_f32sf":
            if self.layout == ops.MASKED:
                return ops.grouped_gemm_f32sf_masked(a, sfa, wq, sfb, b.counts, self.align_or_max_m, d=d,
                                                     expected_m=self.expected_m, flags=self.flags)
            return ops.grouped_gemm_f32sf_contig(a, sfa, wq, sfb, b.seg_start, b.counts, d=d, flags=self.flags)
        if self.fmt == "nvfp4":
            if self.layout == ops.MASKED:
                return ops.grouped_gemm_nvfp4_masked(a, sfa, self.a_exp, wq, sfb, b_exp, b.counts,
                                                     self.align_or_max_m, d=d, expected_m=self.expected_m,
                                                     flags=self.flags)
            return ops.grouped_gemm_nvfp4_contig(a, sfa, self.a_exp, wq, sfb, b_exp, b.seg_start, b.counts, d=d,
                                                 flags=self.flags)
        if self.layout == ops.MASKED:
            return ops.grouped_gemm_masked(a, sfa, wq, sfb, b.counts, self.align_or_max_m, d=d,
                                           expected_m=self.expected_m, flags=self.flags)
        return ops.grouped_gemm_contig(a, sfa, wq, sfb, b.seg_start, b.counts, d=d, flags=self.flags)

    def step(self, x, topk_ids, topk_weights, h2=None, z=None, timer=None):
        """Run the whole path; ``h2`` is the packed bf16 [m_cap, K2] input of the second GEMM;
        the combined output goes to ``z`` (default: this object's output buffer).  Small batches
        quantise, route and scatter in one launch (``dispatch``).  ``timer(name)``, if given, is a
        context manager wrapped around each stage (``dispatch`` or ``quantise`` + ``route``,
        ``gemm``, ``quantise2`` + ``gemm2``, ``combine``), e.g. to record CUDA events."""
        t = timer if timer is not None else _no_timer
        self._stage_in(x, topk_ids, t)
        with t("gemm"):
            self.gemm(self.bufs.a_packed, self.bufs.sfa_packed, self.wq, self.sfb, self.y, self.b_exp)
        out = self.y
        if self.two_gemms and self.fmt == "bf16":
            with t("gemm2"):
                self.gemm(h2, None, self.w2q, None, self.y2)
            out = self.y2
        elif self.two_gemms:
            with t("quantise2"):
                # FP8: only the routed rows of the packed down-projection input (contiguous layout)
                rows = None
                if self.layout == ops.CONTIGUOUS and h2.shape[0] == self.bufs.m_cap:
                    rows = (self.bufs.token_of_row, self.bufs.seg_start[self.E:])
                self._quantise(h2, self.q2, self.sf2, rows=rows)
            with t("gemm2"):
                self.gemm(self.q2, self.sf2, self.w2q, self.sfb2, self.y2, self.b2_exp)
            out = self.y2
        z = self.z if z is None else z
        with t("combine"):
            ops.combine(out, self.bufs.output_index, topk_weights, z=z)
        return z

    def _stage_in(self, x, topk_ids, t):
        """Quantise + route + scatter of the activations into the packed operand."""
        if self.fused_dispatch and self.fmt == "nvfp4":
            with t("dispatch"):
                ops.dispatch_nvfp4(x, topk_ids, self.E, self.layout, self.align_or_max_m, a_exp=self.a_exp,
                                   bufs=self.bufs)
        elif self.fused_dispatch:
            with t("dispatch"):
                ops.dispatch(x, topk_ids, self.E, self.layout, self.align_or_max_m, bufs=self.bufs)
        elif self.route_quantise:
            with t("dispatch"):
                ops.route_quantise(x, topk_ids, self.E, self.layout, self.align_or_max_m, bufs=self.bufs)
        elif self.fmt == "bf16":
            with t("route"):
                ops.route(topk_ids, self.E, self.layout, self.align_or_max_m, q=x, bufs=self.bufs, fmt="bf16")
        else:
            with t("quantise"):
                self._quantise(x, self.q, self.sf)
            with t("route"):
                ops.route(topk_ids, self.E, self.layout, self.align_or_max_m, q=self.q, sf=self.sf, bufs=self.bufs,
                          fmt=self.fmt)

    def capture(self, x, topk_ids, topk_weights, h2=None):
        """Record one step on these (static) input tensors into a CUDA graph.

        Every library call is stream-ordered with no host synchronisation or
        allocation, so the whole step is capturable; a first eager step runs
        before the capture so that one-time set-up (symbol lookups, kernel
        attributes) happens outside it.  ``replay()`` re-runs the step on
        whatever the input tensors hold.
        """
        self.step(x, topk_ids, topk_weights, h2)
        torch.cuda.synchronize()
        # the graph reads these tensors' memory on every replay: keep them alive with it (torch
        # releases cached blocks to the driver when a capture begins, so a dropped input would
        # leave the graph pointing at unmapped memory)
        self._graph_inputs = (x, topk_ids, topk_weights, h2)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.step(x, topk_ids, topk_weights, h2)
        self.graph = graph
        return graph

    def replay(self):
        self.graph.replay()
        return self.z


class HostStreamedPath:
    """Runs a MoEPath over batches held in pinned host memory, overlapping each
    batch's host-to-device copy and the previous result's device-to-host copy
    with the current step's kernels: two device input/output buffer sets, one
    CUDA graph per set, and a copy stream ordered against the compute stream by
    events."""

    def __init__(self, path, T, K, kr, h2=None, device="cuda"):
        self.path = path
        self.sets = []
        for _ in range(2):
            dx = torch.zeros((T, K), dtype=torch.bfloat16, device=device)
            # placeholder routing for the set-up passes: assignments spread evenly over the experts
            dids = (torch.arange(T * kr, dtype=torch.int32, device=device) % path.E).reshape(T, kr)
            dp = torch.full((T, kr), 1.0 / kr, dtype=torch.float32, device=device)
            z = torch.empty_like(path.z)
            path.step(dx, dids, dp, h2, z=z)                 # eager pass: one-time set-up outside the capture
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                path.step(dx, dids, dp, h2, z=z)
            self.sets.append((dx, dids, dp, z, graph))
        self.copy = torch.cuda.Stream(device=device)
        self.h2d_done = [torch.cuda.Event() for _ in range(2)]
        self.comp_done = [torch.cuda.Event() for _ in range(2)]
        self.d2h_done = [torch.cuda.Event() for _ in range(2)]

    def _h2d(self, k, batch):
        dx, dids, dp, _, _ = self.sets[k]
        hx, hids, hp = batch
        dx.copy_(hx, non_blocking=True)
        dids.copy_(hids, non_blocking=True)
        dp.copy_(hp, non_blocking=True)
        self.h2d_done[k].record(self.copy)

    def run(self, host_batches, host_outputs, start_event=None, end_event=None):
        """Process every (x, ids, weights) pinned batch into the matching pinned output."""
        comp = torch.cuda.current_stream()
        n = len(host_batches)
        self.copy.wait_stream(comp)
        with torch.cuda.stream(self.copy):
            if start_event is not None:
                start_event.record(self.copy)
            self._h2d(0, host_batches[0])
        for i in range(n):
            k = i % 2
            comp.wait_event(self.h2d_done[k])
            if i >= 2:
                comp.wait_event(self.d2h_done[k])           # output buffer k was read back
            self.sets[k][4].replay()
            self.comp_done[k].record(comp)
            with torch.cuda.stream(self.copy):
                if i + 1 < n:
                    k2 = (i + 1) % 2
                    if i >= 1:
                        self.copy.wait_event(self.comp_done[k2])   # step i-1 has finished reading input set k2
                    self._h2d(k2, host_batches[i + 1])
                self.copy.wait_event(self.comp_done[k])
                host_outputs[i].copy_(self.sets[k][3], non_blocking=True)
                self.d2h_done[k].record(self.copy)
        if end_event is not None:
            with torch.cuda.stream(self.copy):
                end_event.record(self.copy)
        comp.wait_stream(self.copy)
