"""B300-native (sm_103a) DeepSeekMoE feed-forward layer.

The layer computes h' = u + sum of shared SwiGLU experts + sum of g_i times
the routed SwiGLU experts, with sigmoid affinities, bias-adjusted top-k
selection and gates normalised over the selected experts (DeepSeek-V3
technical report, as read on ai.flicky.cc section 2.1.2 and xyznot.com
Method 2), in bf16 or in the fine-grained FP8 E4M3 scheme (ai.flicky.cc
section 3.3).  Every step runs in libmoe_b300.so (hand-written CUDA for
sm_103a behind the C ABI of include/moe.h); this package only marshals
arguments.
"""
from . import capi
from .capi import (MoEError, moe_bias_update, moe_combine, moe_forward, moe_forward_replicated, moe_grouped_ffn,
                   moe_pack_gate_up, moe_permute, moe_plan_replicas, moe_quantize_fp8_blocks,
                   moe_read_device_status, moe_route, moe_route_noalloc, moe_selftest_wait_timeout,
                   moe_workspace_size)
from .layer import CapturedForward, HostPipeline, MoELayer, ReplicatedExperts

__all__ = ["capi", "CapturedForward", "HostPipeline", "MoEError", "MoELayer", "ReplicatedExperts", "moe_forward_replicated",
           "moe_plan_replicas", "moe_bias_update", "moe_combine", "moe_forward", "moe_grouped_ffn",
           "moe_pack_gate_up", "moe_permute", "moe_quantize_fp8_blocks", "moe_read_device_status", "moe_route",
           "moe_route_noalloc", "moe_selftest_wait_timeout", "moe_workspace_size"]
