"""GB300-native MoE expert-parallel dispatch/combine on one GPU.

The path -- route -> count -> permute/pack -> all-to-all-v dispatch ->
(expert) -> combine -> unpermute with the top-k weighted sum -- runs in the
hand-written sm_103a kernels of ``libmoe_ep.so`` (sources in ``csrc/``, C ABI
in ``include/moe_ep.h``). This package holds the ctypes binding
(``binding``), a buffer-owning convenience layer (``layer``), the seeded
input generators (``workloads``) and byte accounting (``accounting``).
Importing the package does not load the library; the first binding call does,
and fails loudly if the library was not built.
"""
from . import accounting, workloads  # noqa: F401
from .binding import (  # noqa: F401
    MOE_BF16, MOE_FP8_E4M3, MoeError, load_library, make_config, moe_combine,
    moe_dispatch, moe_dispatch_layout, moe_error_string, moe_expert_standin, moe_get_layout,
    moe_handle_create, moe_read_status, moe_recv_rows_max, moe_route_dispatch_layout,
    moe_route_topk, moe_workspace_bytes)
from .build import build  # noqa: F401
from .layer import MoeLayer  # noqa: F401
