"""GB300-native FP8 block-scaled MoE routing + grouped GEMM.

The compute path is ``libbsfroute.so`` (hand-written sm_103a CUDA behind the C
ABI of ``include/bsfroute.h``); this package only builds and binds it.
"""

from .build import build as build_library, LIB_PATH  # noqa: F401
from . import ops  # noqa: F401
from .ops import (  # noqa: F401
    CONTIGUOUS, MASKED, B_HOST_MAPPED, B_TILED, tile_weights, quantise_act, quantise_weight, prepare_weight_sf, route, RouteBuffers,
    route_capacity, dispatch, dispatch_supported, grouped_gemm_contig, grouped_gemm_masked, combine, device_error, sf_ld, sf_words,
)
from .pipeline import MoEPath, HostStreamedPath  # noqa: F401
