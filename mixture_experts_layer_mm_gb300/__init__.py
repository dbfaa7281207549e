"""Fused Mixture-of-Experts layer for one GB300 (sm_103a).

The product is the C-ABI library ``libmm.so`` (include/mm.h); this package
holds its CUDA sources (``csrc/``), the in-tree build (``buildlib``), a thin
ctypes binding with the same entry-point names (``_lib``) and the seeded
synthetic inputs shared with the tests (``synthetic``).
"""
from ._lib import (  # noqa: F401
    FORWARD_BLOCK_M, LIB_PATH, MM_ERR_CUDA, MM_ERR_DEVICE, MM_ERR_INVALID_ARG,
    MM_ERR_NO_MEMORY, MM_ERR_TIMEOUT, MM_ERR_UNSUPPORTED, MM_GEMM_DOWN, MM_GEMM_GATE_UP,
    MM_OK, PROFILE_STAGES, MMError, SIGNATURES, lib, mm_add_rmsnorm, mm_align,
    mm_align_capacity, mm_align_noalloc, mm_gated_mlp, mm_gated_mlp_workspace_size,
    mm_grouped_gemm, mm_moe_forward, mm_moe_forward_add_norm, mm_moe_forward_add_norm_residual,
    mm_moe_forward_partial, mm_moe_forward_profiled, mm_moe_forward_single_launch, mm_round_bf16, tp_slice,
    mm_moe_workspace_layout, mm_moe_workspace_size, forward_routing, WS_LAYOUT_FIELDS,
    mm_poll_device_status, mm_route, mm_selftest_wait_timeout, mm_selftest_layer_barrier_timeout,
    mm_shutdown, status_string,
)
