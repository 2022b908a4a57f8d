"""Routed mixture-of-experts layer (softmax top-k router, NVFP4 experts, fused un-route)
for GB300 (sm_103a): the C-ABI library libroutedmoe.so plus a thin ctypes binding.

High-level use (torch tensors on a CUDA device):

    import routed_moe_decode_gb300 as moe
    layer = moe.MoeLayer(T, d, ffn, E, k)
    out = layer(logits, hidden, weights, residual)     # weights: dict of NVFP4 tensors

The package contains no compute of its own: every step runs in the library's kernels.
"""
from ._lib import (ALGO_AUTO, ALGO_MMA, ALGO_SIMT, ALGO_TCGEN05, ALGO_WIDE, MOE_DEV_BAD_EXPERT_ID, MOE_DEV_H_SATURATED, MOE_DEV_Y_SATURATED,
                   MOE_DEV_HIDDEN_RANGE, MOE_DEV_TIMEOUT, MoeError, Shape, Workspace, auto_algo, check_shape, forward,
                   forward_expert_kernels, forward_experts, forward_prepare, forward_unroute, front,
                   forward_experts_expert_range, layer, layer_expert_range, layer_launches, forward_unroute_gated, layer_expert_scales, layer_from_hidden, layer_gated, lib, plan, plan_expert_range, plan_summary, router_logits, selftest_expert_part, selftest_expert_timeout, plan_views, read_status, route_topk, shape_of, unroute_fused,
                   workspace_bytes)
from ._layer import MoeLayer

__all__ = ["ALGO_AUTO", "ALGO_MMA", "ALGO_SIMT", "ALGO_TCGEN05", "ALGO_WIDE", "MOE_DEV_BAD_EXPERT_ID", "MOE_DEV_H_SATURATED", "MOE_DEV_Y_SATURATED",
           "MOE_DEV_HIDDEN_RANGE", "MOE_DEV_TIMEOUT", "MoeError", "MoeLayer", "Shape", "Workspace",
           "auto_algo", "check_shape", "forward", "forward_expert_kernels", "forward_experts", "forward_prepare", "forward_unroute", "front", "forward_experts_expert_range", "layer", "layer_expert_range", "layer_launches", "forward_unroute_gated", "layer_expert_scales", "layer_from_hidden", "layer_gated", "lib", "plan", "plan_expert_range", "plan_summary", "router_logits", "selftest_expert_part", "selftest_expert_timeout", "plan_views", "read_status",
           "route_topk", "shape_of", "unroute_fused", "workspace_bytes"]
