"""MoE expert-parallel dispatch / combine for one GB300 GPU (sm_103a).

The compute lives in libep_gb300.so (hand-written CUDA behind the C ABI of
include/ep_gb300.h); this package is its thin Python binding plus buffer
management.  Importing the package does not load the library; the first call
does, and raises ImportError when it has not been built.
"""
from ._lib import (EP_ERR_CUDA, EP_ERR_INVALID_ARG, EP_ERR_MISALIGNED, EP_ERR_UNSUPPORTED,
                   EP_ERR_WORKSPACE, EP_OK, EP_QUANT_BF16, EP_QUANT_FP8_E4M3_B128,
                   EP_STATUS_BAD_EXPERT, EP_STATUS_CAPACITY, EPError, ep_combine, ep_dispatch,
                   ep_dispatch_fused, EP_FUSED_MAX_TOKENS, ep_localize_expert_ids,
                   ep_dispatch_layout, ep_dispatch_layout_noalloc, ep_layout_workspace_bytes, ep_max_recv_rows,
                   ep_status_string, load_library, ep_layout_experts_workspace_bytes,
                   ep_dispatch_layout_experts, ep_combine_weighted, ep_selftest_wait_timeout,
                   EP_STATUS_TIMEOUT, ep_cast_transpose_t_bytes, ep_cast_transpose_experts,
                   ep_dispatch_with_layout, ep_dispatch_with_layout_launches,
                   ep_dispatch_experts_with_layout, ep_dispatch_regions, ep_combine_regions,
                   ep_dispatch_regions_with_layout)
from .pipeline import DispatchCombine

__all__ = [
    "EP_OK", "EP_ERR_INVALID_ARG", "EP_ERR_MISALIGNED", "EP_ERR_UNSUPPORTED", "EP_ERR_CUDA",
    "EP_ERR_WORKSPACE", "EP_STATUS_BAD_EXPERT", "EP_STATUS_CAPACITY", "EP_QUANT_BF16",
    "EP_QUANT_FP8_E4M3_B128", "EPError", "ep_dispatch_layout", "ep_dispatch", "ep_combine",
    "ep_dispatch_layout_noalloc", "ep_layout_workspace_bytes", "ep_max_recv_rows", "ep_status_string", "load_library",
    "DispatchCombine", "ep_dispatch_fused", "EP_FUSED_MAX_TOKENS", "ep_localize_expert_ids",
    "ep_layout_experts_workspace_bytes", "ep_dispatch_layout_experts", "ep_combine_weighted",
    "ep_selftest_wait_timeout", "EP_STATUS_TIMEOUT", "ep_cast_transpose_t_bytes",
    "ep_cast_transpose_experts", "ep_dispatch_with_layout",
    "ep_dispatch_with_layout_launches", "ep_dispatch_experts_with_layout",
    "ep_dispatch_regions", "ep_combine_regions", "ep_dispatch_regions_with_layout",
]
