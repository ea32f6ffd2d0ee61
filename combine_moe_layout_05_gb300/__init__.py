"""Single-GPU MoE layout, dispatch and combine for GB300 (sm_103a).

The computation lives in the CUDA library ``libmoe_layout.so`` (C ABI in
``include/moe_layout.h``); this package builds it (``build.build()``) and
binds it with ctypes.  ``workload`` draws seeded synthetic routing inputs and
``experts`` holds the stand-in experts a test or benchmark runs between
dispatch and combine.
"""
from ._binding import (MOE_DEV_ERR_DUPLICATE, MOE_DEV_ERR_EXPERT_RANGE,
                       MOE_DEV_ERR_REGION_OVERFLOW, MOE_DEV_ERR_TIMEOUT,
                       LayoutBuffers, MoeError, declared_functions,
                       library_path, load, moe_combine, moe_combine_fp8,
                       moe_combine_rank_partial,
                       moe_dispatch, moe_dispatch_recv, moe_dispatch_send,
                       moe_layout, moe_layout_dispatch,
                       moe_layout_dispatch_kernels, moe_layout_kernels, moe_layout_static,
                       moe_layout_workspace_bytes,
                       moe_status_string)

__all__ = [
    "MOE_DEV_ERR_DUPLICATE", "MOE_DEV_ERR_EXPERT_RANGE", "MOE_DEV_ERR_REGION_OVERFLOW",
    "MOE_DEV_ERR_TIMEOUT",
    "LayoutBuffers",
    "MoeError", "declared_functions", "library_path", "load", "moe_combine",
    "moe_combine_fp8", "moe_combine_rank_partial",
    "moe_dispatch", "moe_dispatch_recv", "moe_dispatch_send", "moe_layout", "moe_layout_dispatch", "moe_layout_dispatch_kernels", "moe_layout_kernels", "moe_layout_static",
    "moe_layout_workspace_bytes",
    "moe_status_string",
]
