"""GB300-native single-GPU MoE layer: group-limited router, dispatch
permutation, tcgen05 grouped SwiGLU expert FFN, weighted combine.

The compute lives in ``libmoe.so`` (CUDA for sm_103a, C ABI in
``include/moe.h``); this package is its ctypes binding.  Build the library
with ``python -m dispatch_combine_gb300.build``.
"""
from ._lib import (  # noqa: F401
    LIB_PATH,
    MOE_LAYOUT_CONTIGUOUS,
    MOE_LAYOUT_MASKED,
    MOE_OVERFLOW_DROP,
    MOE_OVERFLOW_SECOND_ROUND,
    MOE_SCORE_SIGMOID_BIAS,
    MOE_SCORE_SOFTMAX,
    SIGNATURES,
    STATUS_NAMES,
    MoeShape,
    MoEError,
    Workspace,
    as_shape,
    lib,
    moe_combine,
    moe_dispatch,
    moe_dispatch_capacity,
    moe_dispatch_noalloc,
    moe_eplb_plan,
    moe_expert_capacity,
    moe_expert_down,
    moe_expert_ffn,
    moe_expert_ffn_workspace_size,
    moe_expert_gate_up,
    moe_get_device_status,
    moe_group_topk,
    moe_layer,
    moe_layer_capacity,
    moe_layer_capacity_workspace_size,
    moe_layer_launch_count,
    moe_route,
    moe_route_from_logits,
    moe_selftest_wait_timeout,
    moe_status_string,
    moe_workspace_size,
    shape_struct,
)
