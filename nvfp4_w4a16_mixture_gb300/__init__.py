"""Routed-expert NVFP4 W4A16 MoE block for one GB300 (sm_103a).

The work happens in libflint_moe.so (hand-written CUDA, C ABI in
include/flint_moe.h); this package holds the ctypes binding with the same
names, the in-tree build step and the seeded synthetic-input generator.
"""
from ._lib import (EXPORTED, FLINT_ERR_CUDA, FLINT_ERR_INVALID_ARG, FLINT_ERR_SCRATCH,
                   FLINT_ERR_TIMEOUT, FLINT_ERR_UNSUPPORTED, FLINT_ERR_WORKSPACE,
                   FLINT_FAULT_DOWN_HANDOVER, FLINT_FAULT_NONE, FLINT_OK, FLINT_PATH_DECODE,
                   FLINT_PATH_DECODE_FALLBACK, FLINT_PATH_GROUPED, FLINT_PATH_NONE,
                   FLINT_PATH_SINGLE_LAUNCH,
                   FlintMoEError, alloc_workspace, flint_moe_debug_fault, flint_moe_forward,
                   flint_moe_plan, flint_moe_prefer_path, flint_moe_route,
                   flint_moe_route_noalloc, flint_moe_route_noalloc_bytes,
                   flint_moe_route_noalloc_capacity, flint_moe_status, flint_moe_strerror,
                   flint_moe_workspace_bytes, forward_layer, library_path, load,
                   flint_moe_forward_add_norm, forward_add_norm_layer, flint_moe_record_spans,
                   spans_of, SPAN_NAMES, flint_moe_forward_bf16, flint_moe_forward_nvfp4_shared,
                   flint_qkv_workspace_bytes, flint_qkv_fused)

__all__ = [
    "EXPORTED", "FLINT_OK", "FLINT_ERR_INVALID_ARG", "FLINT_ERR_UNSUPPORTED",
    "FLINT_ERR_WORKSPACE", "FLINT_ERR_CUDA", "FLINT_ERR_TIMEOUT", "FLINT_ERR_SCRATCH",
    "FLINT_FAULT_NONE", "FLINT_FAULT_DOWN_HANDOVER", "FLINT_PATH_NONE", "FLINT_PATH_SINGLE_LAUNCH",
    "FLINT_PATH_DECODE", "FLINT_PATH_DECODE_FALLBACK", "FLINT_PATH_GROUPED", "flint_moe_plan",
    "flint_moe_prefer_path", "flint_moe_forward_add_norm", "forward_add_norm_layer",
    "flint_moe_record_spans", "spans_of", "SPAN_NAMES", "flint_moe_forward_bf16",
    "flint_moe_forward_nvfp4_shared", "flint_qkv_workspace_bytes", "flint_qkv_fused",
    "FlintMoEError", "alloc_workspace", "flint_moe_debug_fault", "flint_moe_forward",
    "flint_moe_route",
    "flint_moe_route_noalloc", "flint_moe_route_noalloc_bytes",
    "flint_moe_route_noalloc_capacity", "flint_moe_status",
    "flint_moe_strerror", "flint_moe_workspace_bytes", "forward_layer", "library_path", "load",
]
