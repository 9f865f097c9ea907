"""ctypes binding of the C ABI in include/moe.h -- argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch
tensors (device memory) or None, passes their data pointers and the current
CUDA stream, and raises MoEError on a non-OK status.  No arithmetic of the
layer happens in Python: every step runs in libmoe_b300.so.  There is no
fallback: if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_B300_LIBRARY=check loads the range-checked build (build.py --check)
LIB_PATH = os.path.join(_PKG, "libmoe_b300_check.so" if os.environ.get("MOE_B300_LIBRARY") == "check"
                        else "libmoe_b300.so")

MOE_BF16, MOE_FP8_E4M3, MOE_FP8_UE8M0 = 0, 1, 2

# Every symbol include/moe.h declares.
EXPORTS = (
    "moe_status_string", "moe_workspace_size", "moe_route", "moe_route_noalloc", "moe_permute", "moe_grouped_ffn",
    "moe_combine", "moe_bias_update", "moe_forward", "moe_forward_profiled", "moe_forward_replicated",
    "moe_plan_replicas", "moe_backward", "moe_backward_workspace_size", "moe_transpose_expert_weights",
    "moe_transpose_expert_weights_fp8",
    "moe_pack_gate_up",
    "moe_quantize_fp8_blocks",
    "moe_read_device_status", "moe_selftest_wait_timeout",
)


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class moe_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("inter", ctypes.c_int32), ("prec", ctypes.c_int32),
                ("route_groups", ctypes.c_int32), ("route_group_limit", ctypes.c_int32)]


class moe_weights_t(ctypes.Structure):
    _fields_ = [("w13t", ctypes.c_void_p), ("w2t", ctypes.c_void_p), ("ws13t", ctypes.c_void_p),
                ("ws2t", ctypes.c_void_p), ("w13t_scale", ctypes.c_void_p), ("w2t_scale", ctypes.c_void_p),
                ("ws13t_scale", ctypes.c_void_p), ("ws2t_scale", ctypes.c_void_p)]


class moe_grads(ctypes.Structure):
    _fields_ = [("du", ctypes.c_void_p), ("dcentroids", ctypes.c_void_p), ("dw13", ctypes.c_void_p),
                ("dw2", ctypes.c_void_p), ("dws13", ctypes.c_void_p), ("dws2", ctypes.c_void_p)]


class moe_weights(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("ws13", ctypes.c_void_p), ("ws13_scale", ctypes.c_void_p),
                ("ws2", ctypes.c_void_p), ("ws2_scale", ctypes.c_void_p), ("centroids", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe_b300.so (build it with mixture_experts_layer_87_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run python -m mixture_experts_layer_87_b300.build)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        D = ctypes.POINTER(moe_dims)
        sig = {
            "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "moe_workspace_size": ([D, ctypes.POINTER(sz)], ctypes.c_int),
            "moe_route": ([D, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "moe_route_noalloc": ([D, vp, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "moe_permute": ([D, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "moe_grouped_ffn": ([D, i32, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "moe_combine": ([D, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "moe_bias_update": ([i32, i32, i32, vp, f32, vp, vp], ctypes.c_int),
            "moe_forward": ([D, ctypes.POINTER(moe_weights), vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "moe_forward_profiled": ([D, ctypes.POINTER(moe_weights), vp, vp, vp, vp, vp, sz, vp,
                                      ctypes.POINTER(vp), i32], ctypes.c_int),
            "moe_forward_replicated": ([D, ctypes.POINTER(moe_weights), vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp],
                                       ctypes.c_int),
            "moe_plan_replicas": ([i32, vp, i32, vp, vp, vp], ctypes.c_int),
            "moe_backward_workspace_size": ([D, ctypes.POINTER(sz)], ctypes.c_int),
            "moe_transpose_expert_weights": ([i32, i32, i32, vp, vp, vp, vp, vp], ctypes.c_int),
            "moe_transpose_expert_weights_fp8": ([i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "moe_backward": ([D, ctypes.POINTER(moe_weights), ctypes.POINTER(moe_weights_t), vp, vp, vp,
                              ctypes.POINTER(moe_grads), vp, sz, vp], ctypes.c_int),
            "moe_pack_gate_up": ([vp, vp, i32, i32, i32, vp, vp], ctypes.c_int),
            "moe_quantize_fp8_blocks": ([vp, i64, i32, vp, vp, i32, vp], ctypes.c_int),
            "moe_read_device_status": ([vp, vp], ctypes.c_int),
            "moe_selftest_wait_timeout": ([vp, sz, i32, vp], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MoEError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    assert isinstance(t, torch.Tensor) and t.is_contiguous(), "tensors must be contiguous"
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return stream


def dims(T, d, E, k, n_shared, inter, prec, route_groups=0, route_group_limit=0) -> moe_dims:
    p = {"bf16": MOE_BF16, "fp8": MOE_FP8_E4M3, "fp8_ue8m0": MOE_FP8_UE8M0}.get(prec, prec)
    return moe_dims(int(T), int(d), int(E), int(k), int(n_shared), int(inter), int(p), int(route_groups),
                    int(route_group_limit))


# ---------------------------------------------------------------- entry points
def moe_workspace_size(dm: moe_dims) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(dm), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_route(dm, u, centroids, bias, topk_idx, topk_gate, counts, ws, stream=None):
    _check(lib().moe_route(ctypes.byref(dm), _ptr(u), _ptr(centroids), _ptr(bias), _ptr(topk_idx), _ptr(topk_gate),
                           _ptr(counts), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_route")


MOE_ROUTE_NOALLOC_MAX_LOGITS = 1 << 21


def moe_route_noalloc(dm, u, centroids, bias, topk_idx, topk_gate, counts, device_status=None, stream=None):
    """moe_route without a workspace, for callers that cannot allocate device
    memory: its logits scratch is a fixed array inside the library (T*E at most
    MOE_ROUTE_NOALLOC_MAX_LOGITS).  device_status: optional int32 device tensor
    of one element that receives the call's device-side status."""
    _check(lib().moe_route_noalloc(ctypes.byref(dm), _ptr(u), _ptr(centroids), _ptr(bias), _ptr(topk_idx),
                                   _ptr(topk_gate), _ptr(counts), _ptr(device_status), _stream(stream)),
           "moe_route_noalloc")


def moe_permute(dm, topk_idx, u, offsets, perm, slot, x_perm, x_scale, ws, stream=None):
    _check(lib().moe_permute(ctypes.byref(dm), _ptr(topk_idx), _ptr(u), _ptr(offsets), _ptr(perm), _ptr(slot),
                             _ptr(x_perm), _ptr(x_scale), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream)), "moe_permute")


def moe_grouped_ffn(dm, n_groups, rows, offsets, x, x_scale, w13, w13_scale, w2, w2_scale, y, ws, stream=None,
                    group_expert=None, n_weight_experts=0):
    _check(lib().moe_grouped_ffn(ctypes.byref(dm), int(n_groups), int(rows), _ptr(offsets), _ptr(group_expert),
                                 int(n_weight_experts), _ptr(x), _ptr(x_scale), _ptr(w13), _ptr(w13_scale), _ptr(w2),
                                 _ptr(w2_scale), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_grouped_ffn")


def moe_combine(dm, u, shared_y, y_perm, slot, topk_gate, out, stream=None):
    _check(lib().moe_combine(ctypes.byref(dm), _ptr(u), _ptr(shared_y), _ptr(y_perm), _ptr(slot), _ptr(topk_gate),
                             _ptr(out), _stream(stream)), "moe_combine")


def moe_bias_update(E, T, k, counts, gamma, bias, stream=None):
    _check(lib().moe_bias_update(int(E), int(T), int(k), _ptr(counts), float(gamma), _ptr(bias), _stream(stream)),
           "moe_bias_update")


def weights_struct(w13, w13_scale, w2, w2_scale, ws13, ws13_scale, ws2, ws2_scale, centroids) -> moe_weights:
    return moe_weights(_ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(ws13), _ptr(ws13_scale),
                       _ptr(ws2), _ptr(ws2_scale), _ptr(centroids))


def moe_forward(dm, weights: moe_weights, u, bias, out, counts_out, ws, stream=None):
    _check(lib().moe_forward(ctypes.byref(dm), ctypes.byref(weights), _ptr(u), _ptr(bias), _ptr(out),
                             _ptr(counts_out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_forward")


def moe_plan_replicas(counts, n_extra):
    """Host plan of n_extra copies of the most loaded experts: (replica_first,
    replica_count, slot_expert) as int32 CPU tensors (counts: CPU int32 [E])."""
    counts = counts.to(torch.int32).contiguous()
    assert not counts.is_cuda
    E = counts.numel()
    first = torch.empty(E, dtype=torch.int32)
    copies = torch.empty(E, dtype=torch.int32)
    slot_expert = torch.empty(E + int(n_extra), dtype=torch.int32)
    _check(lib().moe_plan_replicas(int(E), _ptr(counts), int(n_extra), _ptr(first), _ptr(copies), _ptr(slot_expert)),
           "moe_plan_replicas")
    return first, copies, slot_expert


def moe_forward_replicated(dm, weights: moe_weights, u, bias, replica_first, replica_count, slot_expert, out,
                           counts_out, ws, stream=None):
    _check(lib().moe_forward_replicated(ctypes.byref(dm), ctypes.byref(weights), _ptr(u), _ptr(bias),
                                        _ptr(replica_first), _ptr(replica_count), _ptr(slot_expert),
                                        int(slot_expert.numel()), _ptr(out), _ptr(counts_out), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(stream)), "moe_forward_replicated")


PROFILE_STAGES = ("router_gemm", "topk", "scan_plan", "gather", "routed_gate_up", "routed_down",
                  "shared_gate_up", "shared_down", "combine")
MOE_PROFILE_EVENTS = len(PROFILE_STAGES) + 1


def moe_forward_profiled(dm, weights: moe_weights, u, bias, out, counts_out, ws, events, stream=None):
    """events: MOE_PROFILE_EVENTS torch.cuda.Event(enable_timing=True), already created."""
    handles = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_forward_profiled(ctypes.byref(dm), ctypes.byref(weights), _ptr(u), _ptr(bias), _ptr(out),
                                      _ptr(counts_out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream),
                                      handles, len(events)), "moe_forward_profiled")


def moe_pack_gate_up(w1, w3, E, inter, d, w13, stream=None):
    _check(lib().moe_pack_gate_up(_ptr(w1), _ptr(w3), int(E), int(inter), int(d), _ptr(w13), _stream(stream)),
           "moe_pack_gate_up")


def moe_quantize_fp8_blocks(w, rows, cols, q, scale, stream=None, pow2_scales=False):
    _check(lib().moe_quantize_fp8_blocks(_ptr(w), int(rows), int(cols), _ptr(q), _ptr(scale), int(bool(pow2_scales)),
                                         _stream(stream)),
           "moe_quantize_fp8_blocks")


def moe_read_device_status(ws, stream=None) -> int:
    return lib().moe_read_device_status(_ptr(ws), _stream(stream))


def moe_selftest_wait_timeout(ws, timeout_us, stream=None):
    _check(lib().moe_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), int(timeout_us),
                                           _stream(stream)), "moe_selftest_wait_timeout")


def moe_backward_workspace_size(dm: moe_dims) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_backward_workspace_size(ctypes.byref(dm), ctypes.byref(n)), "moe_backward_workspace_size")
    return n.value


def moe_transpose_expert_weights(n_experts, inter, d, w13, w2, w13t, w2t, stream=None):
    _check(lib().moe_transpose_expert_weights(int(n_experts), int(inter), int(d), _ptr(w13), _ptr(w2), _ptr(w13t),
                                              _ptr(w2t), _stream(stream)), "moe_transpose_expert_weights")


def moe_transpose_expert_weights_fp8(n_experts, inter, d, w13, w13_scale, w2, w2_scale, w13t, w13t_scale, w2t,
                                     w2t_scale, stream=None):
    _check(lib().moe_transpose_expert_weights_fp8(int(n_experts), int(inter), int(d), _ptr(w13), _ptr(w13_scale),
                                                  _ptr(w2), _ptr(w2_scale), _ptr(w13t), _ptr(w13t_scale), _ptr(w2t),
                                                  _ptr(w2t_scale), _stream(stream)), "moe_transpose_expert_weights_fp8")


def moe_backward(dm, weights: moe_weights, weights_t: moe_weights_t, u, bias, dout, grads: moe_grads, ws, stream=None):
    _check(lib().moe_backward(ctypes.byref(dm), ctypes.byref(weights), ctypes.byref(weights_t), _ptr(u), _ptr(bias),
                              _ptr(dout), ctypes.byref(grads), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream)), "moe_backward")
