"""ctypes loader of ``libbsfroute.so`` with the C signatures of ``include/bsfroute.h``.

Loading fails loudly when the library has not been built: there is no other
implementation to fall back to.
"""

import ctypes
import os
import re

from .build import LIB_PATH, ROOT

_c_int = ctypes.c_int
_i64 = ctypes.c_int64
_size = ctypes.c_size_t
_p = ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/bsfroute.h
SIGNATURES = {
    "bsf_status_string": (ctypes.c_char_p, [_c_int]),
    "bsf_version": (_c_int, []),
    "bsf_get_device_error": (_c_int, [ctypes.POINTER(ctypes.c_int32), _c_int, _p]),
    "bsf_quantise_act": (_c_int, [_p, _i64, _i64, _p, _p, _i64, _p]),
    "bsf_quantise_act_rows": (_c_int, [_p, _i64, _i64, _p, _p, _p, _p, _i64, _p]),
    "bsf_quantise_weight": (_c_int, [_p, _i64, _i64, _i64, _p, _p, _p]),
    "bsf_prepare_weight_sf": (_c_int, [_p, _i64, _i64, _i64, _p, _p]),
    "bsf_route_workspace_bytes": (_size, [_i64, _i64, _i64]),
    "bsf_route": (_c_int, [_p, _i64, _i64, _i64, _c_int, _i64, _p, _p, _p, _p, _p, _i64,
                           _p, _p, _i64, _i64, _p, _p, _i64, _p, _size, _p]),
    "bsf_route_no_alloc": (_c_int, [_p, _i64, _i64, _i64, _c_int, _i64, _p, _p, _p, _p, _p, _i64,
                                    _p, _p, _i64, _i64, _p, _p, _i64, _p]),
    "bsf_dispatch": (_c_int, [_p, _i64, _i64, _p, _i64, _i64, _c_int, _i64, _p, _p, _p, _p, _p, _i64,
                              _p, _p, _i64, _p]),
    "bsf_route_quantise": (_c_int, [_p, _i64, _i64, _p, _i64, _i64, _c_int, _i64, _p, _p, _p, _p, _p, _i64,
                                    _p, _p, _i64, _p, _size, _p]),
    "bsf_grouped_gemm_contig": (_c_int, [_p, _p, _i64, _i64, _p, _p, _p, _p, _p, _i64, _i64, _i64, _c_int, _p]),
    "bsf_grouped_gemm_masked": (_c_int, [_p, _p, _i64, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _c_int, _p]),
    "bsf_combine": (_c_int, [_p, _i64, _p, _p, _i64, _i64, _i64, _p, _p]),
    "bsf_checksum_u64": (_c_int, [_p, _size, _c_int, _p, _p]),
    "bsf_tile_weights": (_c_int, [_p, _i64, _i64, _i64, _p, _p]),
    "bsf_route_nvfp4": (_c_int, [_p, _i64, _i64, _i64, _c_int, _i64, _p, _p, _p, _p, _p, _i64,
                                 _p, _p, _i64, _i64, _p, _p, _i64, _p, _size, _p]),
    "bsf_route_bf16": (_c_int, [_p, _i64, _i64, _i64, _c_int, _i64, _p, _p, _p, _p, _p, _i64, _p, _i64, _p, _p,
                                _size, _p]),
    "bsf_grouped_gemm_bf16_contig": (_c_int, [_p, _i64, _p, _p, _p, _p, _i64, _i64, _i64, _c_int, _p]),
    "bsf_grouped_gemm_bf16_masked": (_c_int, [_p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _c_int, _p]),
    "bsf_quantise_act_f32sf": (_c_int, [_p, _i64, _i64, _p, _p, _i64, _p]),
    "bsf_quantise_weight_f32sf": (_c_int, [_p, _i64, _i64, _i64, _p, _p, _p]),
    "bsf_route_f32sf": (_c_int, [_p, _i64, _i64, _i64, _c_int, _i64, _p, _p, _p, _p, _p, _i64,
                                 _p, _p, _i64, _i64, _p, _p, _i64, _p, _size, _p]),
    "bsf_grouped_gemm_f32sf_contig": (_c_int, [_p, _p, _i64, _i64, _p, _p, _p, _p, _p, _i64, _i64, _i64, _c_int,
                                               _p]),
    "bsf_grouped_gemm_f32sf_masked": (_c_int, [_p, _p, _i64, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _c_int,
                                               _p]),
    "bsf_nvfp4_tensor_exponent": (_c_int, [_p, _i64, _i64, _p, _p]),
    "bsf_quantise_act_nvfp4": (_c_int, [_p, _i64, _i64, _c_int, _p, _p, _i64, _p]),
    "bsf_quantise_weight_nvfp4": (_c_int, [_p, _i64, _i64, _i64, _p, _p, _p, _p]),
    "bsf_dispatch_nvfp4": (_c_int, [_p, _i64, _i64, _c_int, _p, _i64, _i64, _c_int, _i64, _p, _p, _p, _p, _p,
                                    _i64, _p, _p, _i64, _p]),
    "bsf_grouped_gemm_nvfp4_contig": (_c_int, [_p, _p, _i64, _i64, _c_int, _p, _p, _p, _p, _p, _p, _i64, _i64,
                                               _i64, _c_int, _p]),
    "bsf_grouped_gemm_nvfp4_masked": (_c_int, [_p, _p, _i64, _c_int, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64,
                                               _i64, _c_int, _p]),
}

_LIB = None


def header_symbols():
    """Function names declared in include/bsfroute.h."""
    with open(os.path.join(ROOT, "include", "bsfroute.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(bsf_[a-z0-9_]+)\s*\(", text)))


def load(path: str = LIB_PATH):
    """Load the library once and attach the C signatures."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


class BsfError(RuntimeError):
    pass


def check(status: int, what: str):
    if status != 0:
        msg = load().bsf_status_string(status).decode()
        raise BsfError(f"{what} failed: {msg} (status {status})")
