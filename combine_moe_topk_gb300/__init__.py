"""GB300-native MoE token path: top-k softmax gating, dispatch layout,
dispatch, combine and their backward duals, behind a C ABI
(``libmoe_gb300.so``, declared in ``include/moe_gb300.h``).

``binding`` holds the ctypes entry points with the C names; ``autograd``
the torch.autograd wrappers and the activation-checkpoint handle recorder;
``workloads`` the seeded synthetic inputs.  The CUDA library is loaded on
first use; there is no CPU fallback.
"""
from .binding import (  # noqa: F401
    Handle,
    MoEError,
    moe_capacity,
    moe_combine,
    moe_combine_bwd,
    moe_debug_hold_layout_tile,
    moe_dispatch,
    moe_dispatch_bwd,
    moe_dispatch_layout,
    moe_dispatch_layout_ex,
    moe_grouped_gemm,
    moe_launch_count,
    moe_status_string,
    moe_topk_gate,
    moe_topk_gate_bwd,
)
