"""Thin torch-facing binding of the C ABI (argument marshalling only).

Every function here allocates its outputs with torch (device memory is the
only thing torch provides), passes raw pointers and the current CUDA stream to
``libbsfroute.so`` and returns the tensors.  All arithmetic runs in the CUDA
kernels.  Names follow the C entry points without the ``bsf_`` prefix.
"""

import ctypes

import torch

from . import _lib

CONTIGUOUS = 0
MASKED = 1
B_HOST_MAPPED = 1
B_TILED = 2              # weights in the layout of tile_weights()
# device error bits (BSF_DEVERR_* in bsfroute.h), read with device_error()
DEVERR_EXPERT_ID = 0x1
DEVERR_MASKED_OVERFLOW = 0x2
DEVERR_TIMEOUT = 0x4
DEVERR_BAD_SCALE = 0x8
DEVERR_SEGMENT = 0x10


def _ptr(t):
    """Device pointer of a CUDA tensor; a host tensor here would be read or written by a kernel
    through an address it cannot use, so it is refused before any library call."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    return ctypes.c_void_p(t.data_ptr())


def _wptr(t, flags):
    """Weights / weight scales: CUDA tensors, or pinned host tensors with B_HOST_MAPPED."""
    if t is None:
        return None
    if flags & B_HOST_MAPPED:
        if t.is_cuda or not t.is_pinned():
            raise ValueError("B_HOST_MAPPED weights must be pinned host tensors (tensor.pin_memory())")
        return ctypes.c_void_p(t.data_ptr())
    return _ptr(t)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def sf_ld(rows: int) -> int:
    """Row stride (int32 words) of a packed MN-major SF tensor: rows rounded up to 4."""
    return (rows + 3) // 4 * 4


def sf_words(K: int) -> int:
    return (K // 128 + 3) // 4


def device_error(clear: bool = True, stream=None) -> int:
    code = ctypes.c_int32(0)
    _lib.check(_lib.load().bsf_get_device_error(ctypes.byref(code), int(clear), _stream(stream)), "get_device_error")
    return code.value


def quantise_act(x, q=None, sf=None, stream=None, rows=None):
    """x bf16 [T, K] -> (q uint8 [T, K], sf int32 [ceil(K/512), sf_ld(T)]).  ``rows`` = (token_of_row,
    rows_used) of a packed operand (a RouteBuffers' token_of_row and seg_start[E:]): only its routed
    rows are quantised, the padding rows of q and sf are left unwritten."""
    T, K = x.shape
    x = x.contiguous()
    if q is None:
        q = torch.empty((T, K), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty((sf_words(K), sf_ld(T)), dtype=torch.int32, device=x.device)
    lib = _lib.load()
    if rows is None:
        _lib.check(lib.bsf_quantise_act(_ptr(x), T, K, _ptr(q), _ptr(sf), sf.shape[1], _stream(stream)),
                   "quantise_act")
    else:
        token_of_row, rows_used = rows
        assert token_of_row.dtype == torch.int32 and token_of_row.numel() >= T and rows_used.dtype == torch.int32
        _lib.check(lib.bsf_quantise_act_rows(_ptr(x), T, K, _ptr(token_of_row), _ptr(rows_used), _ptr(q), _ptr(sf),
                                             sf.shape[1], _stream(stream)), "quantise_act_rows")
    return q, sf


def quantise_weight(w, stream=None):
    """w bf16 [E, N, K] -> (q uint8 [E, N, K], sf128 float32 [E, N/128, K/128])."""
    E, N, K = w.shape
    w = w.contiguous()
    q = torch.empty((E, N, K), dtype=torch.uint8, device=w.device)
    sf128 = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=w.device)
    _lib.check(_lib.load().bsf_quantise_weight(_ptr(w), E, N, K, _ptr(q), _ptr(sf128), _stream(stream)),
               "quantise_weight")
    return q, sf128


def prepare_weight_sf(sf128, K: int, stream=None):
    """sf128 float32 [E, N/128, K/128] -> per-row packed int32 [E, ceil(K/512), N]."""
    E, nb, _ = sf128.shape
    N = nb * 128
    sfb = torch.empty((E, sf_words(K), N), dtype=torch.int32, device=sf128.device)
    _lib.check(_lib.load().bsf_prepare_weight_sf(_ptr(sf128.contiguous()), E, N, K, _ptr(sfb), _stream(stream)),
               "prepare_weight_sf")
    return sfb


def tile_weights(b, stream=None):
    """Weights [E, N, ...] (any dtype; rows of ``row_bytes`` bytes) -> the same bytes tiled
    [E][N/128][row_bytes/128][128][128] for the GEMM flag ``B_TILED``; returned as uint8
    [E, N, row_bytes] so that its shape still names the expert and row counts."""
    E, N = b.shape[0], b.shape[1]
    src = b.contiguous().view(torch.uint8).reshape(E, N, -1)
    out = torch.empty_like(src)
    _lib.check(_lib.load().bsf_tile_weights(_ptr(src), E, N, src.shape[2], _ptr(out), _stream(stream)),
               "tile_weights")
    return out


def route_capacity(T: int, kr: int, E: int, layout: int, align_or_max_m: int) -> int:
    """Worst-case packed row count (no device-to-host sync needed)."""
    if layout == MASKED:
        return E * align_or_max_m
    return T * kr + E * (align_or_max_m - 1)


class RouteBuffers:
    """Preallocated outputs of ``route`` / ``dispatch`` (reused across steps).  ``fmt`` picks the
    packed operand: "fp8" (a_packed [m_cap, K], sfa_packed [ceil(K/512), ld]) or "nvfp4"
    (a_packed [m_cap, K/2], sfa_packed [K/64, ld])."""

    def __init__(self, T, kr, E, layout, align_or_max_m, K=0, device="cuda", scatter=True, fmt="fp8"):
        self.T, self.kr, self.E, self.layout, self.align_or_max_m, self.K = T, kr, E, layout, align_or_max_m, K
        self.m_cap = route_capacity(T, kr, E, layout, align_or_max_m)
        i32 = dict(dtype=torch.int32, device=device)
        self.counts = torch.empty(E, **i32)
        self.seg_start = torch.empty(E + 1, **i32)
        self.output_index = torch.empty((T, kr), **i32)
        self.token_of_row = torch.empty(max(self.m_cap, 1), **i32)
        self.m_indices = torch.empty(max(self.m_cap, 1), **i32)
        ws = _lib.load().bsf_route_workspace_bytes(T, kr, E)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        self.fmt = fmt
        if scatter and K and fmt == "fp8_f32sf":
            self.a_packed = torch.empty((max(self.m_cap, 1), K), dtype=torch.uint8, device=device)
            self.sfa_packed = torch.empty((K // 128, sf_ld(self.m_cap)), dtype=torch.float32, device=device)
        elif scatter and K and fmt == "bf16":
            self.a_packed = torch.empty((max(self.m_cap, 1), K), dtype=torch.bfloat16, device=device)
            self.sfa_packed = None
        elif scatter and K and fmt == "nvfp4":
            self.a_packed = torch.empty((max(self.m_cap, 1), K // 2), dtype=torch.uint8, device=device)
            self.sfa_packed = torch.empty((K // 64, sf_ld(self.m_cap)), dtype=torch.int32, device=device)
        elif scatter and K:
            self.a_packed = torch.empty((max(self.m_cap, 1), K), dtype=torch.uint8, device=device)
            self.sfa_packed = torch.empty((sf_words(K), sf_ld(self.m_cap)), dtype=torch.int32, device=device)
        else:
            self.a_packed = self.sfa_packed = None


def route(topk_ids, E, layout, align_or_max_m, q=None, sf=None, bufs=None, stream=None, fmt="fp8"):
    """Routing + optional scatter of quantised rows (``fmt`` "fp8" or "nvfp4") or of bf16 rows
    (``fmt`` "bf16", ``q`` the bf16 activations, no ``sf``); returns a RouteBuffers."""
    T, kr = topk_ids.shape
    K = (q.shape[1] * (2 if fmt == "nvfp4" else 1)) if q is not None else 0
    if bufs is None:
        bufs = RouteBuffers(T, kr, E, layout, align_or_max_m, K=K, device=topk_ids.device, scatter=q is not None,
                            fmt=fmt)
    lib = _lib.load()
    if fmt == "bf16":
        _lib.check(lib.bsf_route_bf16(
            _ptr(topk_ids.contiguous()), T, kr, E, layout, align_or_max_m,
            _ptr(bufs.counts), _ptr(bufs.seg_start), _ptr(bufs.output_index), _ptr(bufs.token_of_row),
            _ptr(bufs.m_indices), bufs.m_cap, _ptr(q.contiguous() if q is not None else None), K,
            _ptr(bufs.a_packed) if q is not None else None, _ptr(bufs.workspace), bufs.workspace.numel(),
            _stream(stream)), "route_bf16")
        return bufs
    fn = {"nvfp4": lib.bsf_route_nvfp4, "fp8_f32sf": lib.bsf_route_f32sf}.get(fmt, lib.bsf_route)
    _lib.check(fn(
        _ptr(topk_ids.contiguous()), T, kr, E, layout, align_or_max_m,
        _ptr(bufs.counts), _ptr(bufs.seg_start), _ptr(bufs.output_index), _ptr(bufs.token_of_row),
        _ptr(bufs.m_indices), bufs.m_cap,
        _ptr(q), _ptr(sf), sf.shape[1] if sf is not None else 0, K,
        _ptr(bufs.a_packed) if q is not None else None, _ptr(bufs.sfa_packed) if q is not None else None,
        bufs.sfa_packed.shape[1] if (q is not None and bufs.sfa_packed is not None) else 0,
        _ptr(bufs.workspace), bufs.workspace.numel(), _stream(stream)), "route")
    return bufs


DISPATCH_MAX_ASSIGNMENTS = 16384
DISPATCH_MAX_EXPERTS = 256


def dispatch_supported(T, kr, E):
    return T * kr <= DISPATCH_MAX_ASSIGNMENTS and E <= DISPATCH_MAX_EXPERTS


def dispatch(x, topk_ids, E, layout, align_or_max_m, bufs=None, stream=None):
    """Quantise + route + scatter in one launch (small batches); returns a RouteBuffers."""
    T, K = x.shape
    kr = topk_ids.shape[1]
    if bufs is None:
        bufs = RouteBuffers(T, kr, E, layout, align_or_max_m, K=K, device=x.device)
    _lib.check(_lib.load().bsf_dispatch(
        _ptr(x.contiguous()), T, K, _ptr(topk_ids.contiguous()), kr, E, layout, align_or_max_m,
        _ptr(bufs.counts), _ptr(bufs.seg_start), _ptr(bufs.output_index), _ptr(bufs.token_of_row),
        _ptr(bufs.m_indices), bufs.m_cap, _ptr(bufs.a_packed), _ptr(bufs.sfa_packed), bufs.sfa_packed.shape[1],
        _stream(stream)), "dispatch")
    return bufs


def route_quantise_supported(kr):
    return kr <= 32


def route_quantise(x, topk_ids, E, layout, align_or_max_m, bufs=None, stream=None):
    """Quantise + route + scatter for batches of any size (routing kernels, then each token's row
    quantised once and written to its k_r packed rows); returns a RouteBuffers."""
    T, K = x.shape
    kr = topk_ids.shape[1]
    if bufs is None:
        bufs = RouteBuffers(T, kr, E, layout, align_or_max_m, K=K, device=x.device)
    _lib.check(_lib.load().bsf_route_quantise(
        _ptr(x.contiguous()), T, K, _ptr(topk_ids.contiguous()), kr, E, layout, align_or_max_m,
        _ptr(bufs.counts), _ptr(bufs.seg_start), _ptr(bufs.output_index), _ptr(bufs.token_of_row),
        _ptr(bufs.m_indices), bufs.m_cap, _ptr(bufs.a_packed), _ptr(bufs.sfa_packed), bufs.sfa_packed.shape[1],
        _ptr(bufs.workspace), bufs.workspace.numel(), _stream(stream)), "route_quantise")
    return bufs


def grouped_gemm_contig(a, sfa, b, sfb, seg_start, counts, d=None, flags=0, stream=None):
    """a uint8 [m_cap, K], b uint8 [E, N, K] -> d bf16 [m_cap, N] (segment rows written)."""
    m_cap, K = a.shape
    E, N, _ = b.shape
    if d is None:
        d = torch.empty((m_cap, N), dtype=torch.bfloat16, device=a.device)
    _lib.check(_lib.load().bsf_grouped_gemm_contig(
        _ptr(a), _ptr(sfa), sfa.shape[1], m_cap, _wptr(b, flags), _wptr(sfb, flags), _ptr(d), _ptr(seg_start), _ptr(counts),
        E, N, K, flags, _stream(stream)), "grouped_gemm_contig")
    return d


def grouped_gemm_masked(a, sfa, b, sfb, masked_m, max_m, d=None, expected_m=0, flags=0, stream=None):
    """a uint8 [E*max_m, K] (or [E, max_m, K]), b uint8 [E, N, K] -> d bf16 [E*max_m, N]."""
    K = a.shape[-1]
    E, N, _ = b.shape
    if d is None:
        d = torch.empty((E * max_m, N), dtype=torch.bfloat16, device=a.device)
    _lib.check(_lib.load().bsf_grouped_gemm_masked(
        _ptr(a), _ptr(sfa), sfa.shape[1], _wptr(b, flags), _wptr(sfb, flags), _ptr(d), _ptr(masked_m), E, max_m, N, K,
        expected_m, flags, _stream(stream)), "grouped_gemm_masked")
    return d


def combine(y, output_index, topk_weights, z=None, stream=None):
    """y bf16 [rows, N] -> z bf16 [T, N]."""
    rows, N = y.shape
    T, kr = output_index.shape
    if z is None:
        z = torch.empty((T, N), dtype=torch.bfloat16, device=y.device)
    _lib.check(_lib.load().bsf_combine(
        _ptr(y), rows, _ptr(output_index.contiguous()), _ptr(topk_weights.contiguous()), T, kr, N, _ptr(z),
        _stream(stream)), "combine")
    return z


def checksum_u64(t, host_mapped=False, out=None, stream=None):
    """XOR of the 64-bit words of a tensor's bytes (device tensor, or pinned host tensor if host_mapped)."""
    nbytes = t.numel() * t.element_size()
    if out is None:
        out = torch.empty(1, dtype=torch.int64, device="cuda")
    _lib.check(_lib.load().bsf_checksum_u64(_wptr(t, B_HOST_MAPPED if host_mapped else 0), nbytes,
                                            B_HOST_MAPPED if host_mapped else 0, _ptr(out),
                                            _stream(stream)), "checksum_u64")
    return out


# ----------------------------------------------------------------------------- NVFP4
def nvfp4_tensor_exponent(x, groups=1, out=None, stream=None):
    """Least j per group with max|x| <= 6 * 448 * 2**j; x bf16 split into ``groups`` equal groups."""
    x = x.contiguous()
    if out is None:
        out = torch.empty(groups, dtype=torch.int32, device=x.device)
    _lib.check(_lib.load().bsf_nvfp4_tensor_exponent(_ptr(x), groups, x.numel() // groups, _ptr(out),
                                                     _stream(stream)), "nvfp4_tensor_exponent")
    return out


def quantise_act_nvfp4(x, a_exp=0, q=None, sf=None, stream=None):
    """x bf16 [T, K] -> (q uint8 [T, K/2], sf int32 [K/64, sf_ld(T)])."""
    T, K = x.shape
    if q is None:
        q = torch.empty((T, K // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty((K // 64, sf_ld(T)), dtype=torch.int32, device=x.device)
    _lib.check(_lib.load().bsf_quantise_act_nvfp4(_ptr(x.contiguous()), T, K, int(a_exp), _ptr(q), _ptr(sf),
                                                  sf.shape[1], _stream(stream)), "quantise_act_nvfp4")
    return q, sf


def quantise_weight_nvfp4(w, b_exp=None, stream=None):
    """w bf16 [E, N, K] -> (q uint8 [E, N, K/2], sfb int32 [E, K/64, N], b_exp int32 [E]).
    Without ``b_exp`` each expert takes its least tensor exponent (``nvfp4_tensor_exponent``)."""
    E, N, K = w.shape
    w = w.contiguous()
    if b_exp is None:
        b_exp = nvfp4_tensor_exponent(w, groups=E, stream=stream)
    q = torch.empty((E, N, K // 2), dtype=torch.uint8, device=w.device)
    sfb = torch.empty((E, K // 64, N), dtype=torch.int32, device=w.device)
    _lib.check(_lib.load().bsf_quantise_weight_nvfp4(_ptr(w), E, N, K, _ptr(b_exp), _ptr(q), _ptr(sfb),
                                                     _stream(stream)), "quantise_weight_nvfp4")
    return q, sfb, b_exp


def dispatch_nvfp4(x, topk_ids, E, layout, align_or_max_m, a_exp=0, bufs=None, stream=None):
    """NVFP4 quantise + route + scatter in one launch (small batches); returns a RouteBuffers."""
    T, K = x.shape
    kr = topk_ids.shape[1]
    if bufs is None:
        bufs = RouteBuffers(T, kr, E, layout, align_or_max_m, K=K, device=x.device, fmt="nvfp4")
    _lib.check(_lib.load().bsf_dispatch_nvfp4(
        _ptr(x.contiguous()), T, K, int(a_exp), _ptr(topk_ids.contiguous()), kr, E, layout, align_or_max_m,
        _ptr(bufs.counts), _ptr(bufs.seg_start), _ptr(bufs.output_index), _ptr(bufs.token_of_row),
        _ptr(bufs.m_indices), bufs.m_cap, _ptr(bufs.a_packed), _ptr(bufs.sfa_packed), bufs.sfa_packed.shape[1],
        _stream(stream)), "dispatch_nvfp4")
    return bufs


def grouped_gemm_nvfp4_contig(a, sfa, a_exp, b, sfb, b_exp, seg_start, counts, d=None, flags=0, stream=None):
    """a uint8 [m_cap, K/2], b uint8 [E, N, K/2] -> d bf16 [m_cap, N] (segment rows written)."""
    m_cap, K2 = a.shape
    E, N, _ = b.shape
    if d is None:
        d = torch.empty((m_cap, N), dtype=torch.bfloat16, device=a.device)
    _lib.check(_lib.load().bsf_grouped_gemm_nvfp4_contig(
        _ptr(a), _ptr(sfa), sfa.shape[1], m_cap, int(a_exp), _wptr(b, flags), _wptr(sfb, flags), _ptr(b_exp), _ptr(d),
        _ptr(seg_start), _ptr(counts), E, N, 2 * K2, flags, _stream(stream)), "grouped_gemm_nvfp4_contig")
    return d


def grouped_gemm_nvfp4_masked(a, sfa, a_exp, b, sfb, b_exp, masked_m, max_m, d=None, expected_m=0, flags=0,
                              stream=None):
    """a uint8 [E*max_m, K/2], b uint8 [E, N, K/2] -> d bf16 [E*max_m, N]."""
    K2 = a.shape[-1]
    E, N, _ = b.shape
    if d is None:
        d = torch.empty((E * max_m, N), dtype=torch.bfloat16, device=a.device)
    _lib.check(_lib.load().bsf_grouped_gemm_nvfp4_masked(
        _ptr(a), _ptr(sfa), sfa.shape[1], int(a_exp), _wptr(b, flags), _wptr(sfb, flags), _ptr(b_exp), _ptr(d), _ptr(masked_m),
        E, max_m, N, 2 * K2, expected_m, flags, _stream(stream)), "grouped_gemm_nvfp4_masked")
    return d


# ----------------------------------------------------------------------------- BF16
def grouped_gemm_bf16_contig(a, b, seg_start, counts, d=None, flags=0, stream=None):
    """a bf16 [m_cap, K], b bf16 [E, N, K] -> d bf16 [m_cap, N] (segment rows written)."""
    m_cap, K = a.shape
    E, N, _ = b.shape
    if d is None:
        d = torch.empty((m_cap, N), dtype=torch.bfloat16, device=a.device)
    _lib.check(_lib.load().bsf_grouped_gemm_bf16_contig(
        _ptr(a), m_cap, _wptr(b, flags), _ptr(d), _ptr(seg_start), _ptr(counts), E, N, K, flags, _stream(stream)),
        "grouped_gemm_bf16_contig")
    return d


def grouped_gemm_bf16_masked(a, b, masked_m, max_m, d=None, expected_m=0, flags=0, stream=None):
    """a bf16 [E*max_m, K], b bf16 [E, N, K] -> d bf16 [E*max_m, N]."""
    K = a.shape[-1]
    E, N, _ = b.shape
    if d is None:
        d = torch.empty((E * max_m, N), dtype=torch.bfloat16, device=a.device)
    _lib.check(_lib.load().bsf_grouped_gemm_bf16_masked(
        _ptr(a), _wptr(b, flags), _ptr(d), _ptr(masked_m), E, max_m, N, K, expected_m, flags, _stream(stream)),
        "grouped_gemm_bf16_masked")
    return d


# ----------------------------------------------------------------------------- FP8 with float32 scales
def quantise_act_f32sf(x, q=None, sf=None, stream=None):
    """x bf16 [T, K] -> (q uint8 [T, K], sf float32 [K/128, sf_ld(T)])."""
    T, K = x.shape
    if q is None:
        q = torch.empty((T, K), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty((K // 128, sf_ld(T)), dtype=torch.float32, device=x.device)
    _lib.check(_lib.load().bsf_quantise_act_f32sf(_ptr(x.contiguous()), T, K, _ptr(q), _ptr(sf), sf.shape[1],
                                                  _stream(stream)), "quantise_act_f32sf")
    return q, sf


def quantise_weight_f32sf(w, stream=None):
    """w bf16 [E, N, K] -> (q uint8 [E, N, K], sf float32 [E, N/128, K/128])."""
    E, N, K = w.shape
    q = torch.empty((E, N, K), dtype=torch.uint8, device=w.device)
    sf = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=w.device)
    _lib.check(_lib.load().bsf_quantise_weight_f32sf(_ptr(w.contiguous()), E, N, K, _ptr(q), _ptr(sf),
                                                     _stream(stream)), "quantise_weight_f32sf")
    return q, sf


def grouped_gemm_f32sf_contig(a, sfa, b, sfb, seg_start, counts, d=None, flags=0, stream=None):
    """a uint8 [m_cap, K], sfa float32 [K/128, ld], b uint8 [E, N, K], sfb float32 [E, N/128, K/128]."""
    m_cap, K = a.shape
    E, N, _ = b.shape
    if d is None:
        d = torch.empty((m_cap, N), dtype=torch.bfloat16, device=a.device)
    _lib.check(_lib.load().bsf_grouped_gemm_f32sf_contig(
        _ptr(a), _ptr(sfa), sfa.shape[1], m_cap, _wptr(b, flags), _wptr(sfb, flags), _ptr(d), _ptr(seg_start), _ptr(counts),
        E, N, K, flags, _stream(stream)), "grouped_gemm_f32sf_contig")
    return d


def grouped_gemm_f32sf_masked(a, sfa, b, sfb, masked_m, max_m, d=None, expected_m=0, flags=0, stream=None):
    """a uint8 [E*max_m, K], sfa float32 [K/128, ld] -> d bf16 [E*max_m, N]."""
    K = a.shape[-1]
    E, N, _ = b.shape
    if d is None:
        d = torch.empty((E * max_m, N), dtype=torch.bfloat16, device=a.device)
    _lib.check(_lib.load().bsf_grouped_gemm_f32sf_masked(
        _ptr(a), _ptr(sfa), sfa.shape[1], _wptr(b, flags), _wptr(sfb, flags), _ptr(d), _ptr(masked_m), E, max_m, N, K, expected_m,
        flags, _stream(stream)), "grouped_gemm_f32sf_masked")
    return d
