"""GB300-native MoE expert-parallel route / layout / dispatch / combine.

The compute path is libep_gb300.so (hand-written CUDA for sm_103a, C ABI in
include/ep.h); ``ep`` is its thin Python binding and ``workloads`` the seeded
synthetic inputs.
"""
from .ep import (EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3_B128, EP_LAYOUT_CONTIG, EP_LAYOUT_MASKED,
                 EPError, Layout, alloc_layout, ep_combine, ep_dispatch, ep_dispatch_layout,
                 ep_dispatch_layout_workspace_size, ep_expert_balance_map,
                 ep_kernel_launch_count, ep_route_dispatch, ep_route_dispatch_workspace_size,
                 ep_route_layout, ep_route_layout_workspace_size, ep_route_topk,
                 ep_selftest_wait_timeout)

__all__ = [
    "EP_DTYPE_BF16", "EP_DTYPE_FP8_E4M3_B128", "EP_LAYOUT_CONTIG", "EP_LAYOUT_MASKED", "EPError",
    "Layout", "alloc_layout", "ep_combine", "ep_dispatch", "ep_dispatch_layout",
    "ep_dispatch_layout_workspace_size", "ep_expert_balance_map", "ep_kernel_launch_count",
    "ep_route_dispatch", "ep_route_dispatch_workspace_size", "ep_route_layout", "ep_route_layout_workspace_size", "ep_route_topk",
    "ep_selftest_wait_timeout",
]
