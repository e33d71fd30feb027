"""ctypes declarations of libgbmoe.so (the C ABI in include/gbmoe.h)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgbmoe.so")

c_i32, c_i64, c_f32, c_sz, c_vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                   ctypes.c_size_t, ctypes.c_void_p)
P_i32 = ctypes.POINTER(ctypes.c_int32)


class ForwardOpts(ctypes.Structure):
    _fields_ = [("reduce_mode", ctypes.c_int32), ("apply_router_weight_on_input", ctypes.c_int32),
                ("expert_map", ctypes.c_void_p), ("num_global_experts", ctypes.c_int32)]


class Fp8Weights(ctypes.Structure):
    _fields_ = [("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("scale_mode", ctypes.c_int32)]


class WqWeights(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w13_scale", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p),
                ("w13_zero", ctypes.c_void_p), ("w2_zero", ctypes.c_void_p)]


class HostIo(ctypes.Structure):
    _fields_ = [("h_hidden", ctypes.c_void_p), ("h_logits", ctypes.c_void_p),
                ("h_out", ctypes.c_void_p), ("d_hidden", ctypes.c_void_p),
                ("d_logits", ctypes.c_void_p), ("topk_weights", ctypes.c_void_p),
                ("topk_ids", ctypes.c_void_p), ("d_out", ctypes.c_void_p)]


class RouteParams(ctypes.Structure):
    _fields_ = [("top_k", ctypes.c_int32), ("routing_method", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("k_group", ctypes.c_int32),
                ("group_count", ctypes.c_int32), ("group_select_mode", ctypes.c_int32),
                ("routed_scaling_factor", ctypes.c_float)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


# name -> (restype, argtypes)
SIGNATURES = {
    "moe_abi_version": (c_i32, []),
    "moe_status_string": (ctypes.c_char_p, [c_i32]),
    "moe_last_error_detail": (ctypes.c_char_p, []),
    "moe_launch_count": (c_i64, []),
    "moe_route": (c_i32, [c_vp, c_i64, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_f32,
                          c_vp, c_vp, c_vp]),
    "moe_route_bf16": (c_i32, [c_vp, c_i64, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                               c_f32, c_vp, c_vp, c_vp]),
    "moe_router_logits": (c_i32, [c_vp, c_vp, c_vp, c_i64, c_i32, c_i32, c_vp, c_vp]),
    "moe_forward_opts": (c_i32, [c_vp, c_vp, c_vp, c_i64, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp,
                                 c_vp, c_vp, c_vp, c_sz, ctypes.POINTER(ForwardOpts), c_vp,
                                 c_vp]),
    "moe_workspace_size_fp8": (c_i32, [c_i64, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_sz)]),
    "moe_forward_fp8": (c_i32, [c_vp, c_vp, c_vp, c_i64, c_i32, c_i32, c_i32, c_i32,
                                ctypes.POINTER(Fp8Weights), c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "moe_quant_rows_fp8": (c_i32, [c_vp, c_i64, c_i32, c_vp, c_vp, c_vp]),
    "moe_dequant_weights": (c_i32, [c_i32, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp,
                                    c_vp]),
    "moe_set_gather_mode": (c_i32, [c_i32]),
    "moe_forward_host": (c_i32, [c_vp, c_i64, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                                 c_vp, ctypes.c_size_t, c_i32, c_vp]),
    "moe_forward_wq": (c_i32, [c_vp, c_vp, c_vp, c_i64, c_i32, c_i32, c_i32, c_i32,
                               ctypes.POINTER(WqWeights), c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "moe_align_capacity": (c_sz, [c_i64, c_i32, c_i32, c_i32]),
    "moe_align_scratch_size": (c_sz, [c_i64, c_i32, c_i32]),
    "moe_align": (c_i32, [c_vp, c_i64, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz,
                          c_vp, c_vp]),
    "moe_align_static_scratch": (c_i32, [c_vp, c_i64, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp,
                                         c_vp, c_vp, c_vp]),
    "moe_workspace_size": (c_i32, [c_i64, c_i32, c_i32, c_i32, c_i32, c_i32,
                                   ctypes.POINTER(c_sz)]),
    "moe_forward": (c_i32, [c_vp, c_vp, c_vp, c_i64, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp,
                            c_vp, c_vp, c_vp, c_sz, c_i32, c_vp, c_vp]),
    "moe_batched_workspace_size": (c_i32, [c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_sz)]),
    "moe_forward_batched": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp,
                                    c_vp, c_vp, c_vp, c_sz, c_vp, c_vp]),
    "moe_workspace_error_word": (c_vp, [c_vp]),
    "moe_read_error": (c_i32, [c_vp, c_i32, c_vp]),
    "moe_workspace_layout": (c_i32, [c_i64, c_i32, c_i32, c_i32, c_i32,
                                     ctypes.POINTER(c_sz)]),
    "moe_selftest_wait_timeout": (c_i32, [c_vp, ctypes.c_uint32, c_vp]),
    "moe_set_gemm_tiles": (c_i32, [c_i32]),
    "moe_set_pdl": (c_i32, [c_i32]),
    "moe_set_wq_decode": (c_i32, [c_i32]),
    "moe_set_item_rows": (c_i32, [c_i32]),
    "moe_set_host_out_direct": (c_i32, [c_i32]),
    "moe_set_small_path": (c_i32, [c_i32]),
    "moe_profiler_start": (c_i32, []),
    "moe_profiler_stop": (c_i32, [ctypes.POINTER(KernelTime), c_i32, P_i32]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libgbmoe.so; raises if it has not been built.  There is no
    fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
            " (there is no CPU or Python fallback for the fused MoE path)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
