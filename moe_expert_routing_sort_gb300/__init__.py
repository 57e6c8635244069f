"""GB300-native (sm_103a) MoE route-sort: router logits -> expert-grouped dispatch metadata.

The compute path is the CUDA library ``libmoe_route_sort.so`` (C ABI in
``include/moe_route_sort.h``); this package holds its thin ctypes binding, the build script
and the seeded input generator used by the tests and the benchmark.
"""
from . import datagen  # noqa: F401
from ._build import build  # noqa: F401
from .binding import (  # noqa: F401
    DEBUG_CLUSTER_TOKENS,
    DEBUG_FORCE_PROXY_FAIL,
    DEBUG_GRID_TOKENS,
    DEBUG_WARP_GRID_TOKENS,
    DEBUG_WAIT_LIMIT_NS,
    DEVICE_BAD_EXPERT_ID,
    RouteSortBuffers,
    RouteSortError,
    library_path,
    gate_route_sort,
    load,
    map_host,
    moe_gate_route_sort,
    moe_route_sort,
    moe_route_sort_debug_set,
    moe_route_sort_noalloc,
    moe_route_sort_noalloc_status,
    moe_route_sort_proxy_selftest,
    moe_route_sort_proxy_state,
    moe_route_sort_softmax,
    moe_route_sort_workspace_bytes,
    moe_sort,
    moe_sort_max_blocks,
    moe_sort_max_padded,
    moe_topk,
    route_sort,
    route_sort_from_host,
    route_sort_mapped,
    route_sort_softmax,
    strerror,
)
