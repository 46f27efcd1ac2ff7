"""ctypes binding of libmoe_w4a16.so (include/moe_w4a16.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions carry the C entry points' names and take torch tensors
(device memory) or plain numbers; errors raise MoeError.  There is no CPU
fallback: without the built library, loading raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_w4a16.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe_w4a16.h")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_MISALIGNED = 3
MOE_ERR_WORKSPACE_TOO_SMALL = 4
MOE_ERR_CUDA = 5
MOE_ERR_DEVICE_TIMEOUT = 6
MOE_PROJ_GATE_UP = 0
MOE_PROJ_DOWN = 1


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32)]


class W4(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("global_scale", ctypes.c_void_p)]


class W4N(ctypes.Structure):
    """Natural-layout NVFP4 weights (the W4A4 entry points)."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("global_scale", ctypes.c_void_p)]


_lib = None
P = ctypes.c_void_p
SZ = ctypes.c_size_t
I32 = ctypes.c_int32
INT = ctypes.c_int

_SIGS = {
    "moe_packed_w4_bytes": (SZ, [I32, I32, I32]),
    "moe_prepack_w4": (INT, [P, P, I32, I32, I32, I32, P, P]),
    "moe_workspace_bytes": (SZ, [Dims]),
    "moe_layer_kernel_launches": (ctypes.c_int, [Dims]),
    "moe_layer_projections_fused": (ctypes.c_int, [Dims]),
    "moe_stage_workspace_bytes": (SZ, [Dims]),
    "moe_router_logits": (INT, [P, P, P, Dims, P, P]),
    "moe_route_topk": (INT, [P, Dims, P, P, P]),
    "moe_permute": (INT, [P, P, Dims, P, P, P, P, P, P, SZ, P]),
    "moe_permute_noalloc": (INT, [P, P, Dims, P, P, P, P, P, P]),
    "moe_w4a16_gate_up_swiglu": (INT, [P, P, W4, Dims, P, P, SZ, P]),
    "moe_w4a16_down": (INT, [P, P, W4, Dims, P, P, SZ, P]),
    "moe_unpermute_combine": (INT, [P, P, P, Dims, P, P]),
    "moe_layer_forward": (INT, [P, P, W4, W4, Dims, P, P, P, P, SZ, P]),
    "moe_layer_forward_profiled": (INT, [P, P, W4, W4, Dims, P, P, P, P, SZ, P, P]),
    "moe_layer_forward_host": (INT, [P, P, W4, W4, Dims, P, P, SZ, P]),
    "moe_host_plan_create": (INT, [P, P, W4, W4, Dims, P, P, SZ, P, ctypes.POINTER(ctypes.c_void_p)]),
    "moe_host_plan_run": (INT, [P]),
    "moe_host_plan_destroy": (INT, [P]),
    "moe_layer_forward_router": (INT, [P, P, P, W4, W4, Dims, P, P, P, P, P, SZ, P]),
    "moe_layer_forward_shared": (INT, [P, P, P, P, W4, W4, W4, W4, Dims, P, P, P, P, P, SZ, P]),
    "moe_get_device_status": (INT, [P, P]),
    "moe_status_string": (ctypes.c_char_p, [INT]),
    "moe_debug_dequant_table": (INT, [P, P]),
    "moe_debug_timeout_probe": (INT, [P, ctypes.c_uint64, P]),
    "moe_debug_counter_timeout_probe": (INT, [P, ctypes.c_uint64, P]),
    "moe_debug_stream_read": (INT, [P, SZ, P, P]),
    "moe_w4a4_workspace_bytes": (SZ, [Dims]),
    "moe_w4a4_kernel_launches": (ctypes.c_int, [Dims]),
    "moe_layer_forward_w4a4": (INT, [P, P, W4N, W4N, Dims, P, P, P, P, SZ, P]),
    "moe_layer_forward_w4a4_profiled": (INT, [P, P, W4N, W4N, Dims, P, P, P, P, SZ, P, P]),
    "moe_quantize_nvfp4": (INT, [P, P, I32, I32, P, P, P]),
    "moe_quantize_nvfp4_f32": (INT, [P, P, I32, I32, P, P, P]),
    "moe_debug_w4a4_gemm": (INT, [I32, P, P, P, W4N, Dims, P, P, P, P]),
    "moe_debug_layer_forward_config": (INT, [P, P, W4, W4, Dims, P, P, P, P, SZ, I32, I32, P, P]),
}


def load(path: str | None = None):
    """Load the shared library (building nothing).  Raises if it is missing."""
    global _lib
    if _lib is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libmoe_w4a16.so not built at {p}; run moe_layer_bit_gb300.build.build()")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols():
    return list(_SIGS)


def status_string(status: int) -> str:
    try:
        return load().moe_status_string(int(status)).decode()
    except RuntimeError:
        return str(status)


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _p(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return ctypes.c_void_p(t.data_ptr())
    return ctypes.c_void_p(int(t))


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def dims(T, H, I, E, k) -> Dims:
    return Dims(int(T), int(H), int(I), int(E), int(k))


def w4(packed: torch.Tensor, global_scale: torch.Tensor) -> W4:
    return W4(packed.data_ptr(), global_scale.data_ptr())


# --------------------------------------------------------------- entry points
def moe_packed_w4_bytes(E, N, K) -> int:
    return int(load().moe_packed_w4_bytes(E, N, K))


def moe_prepack_w4(codes, scales, E, N, K, proj, packed, stream=None):
    _check(load().moe_prepack_w4(_p(codes), _p(scales), E, N, K, proj, _p(packed), _s(stream)), "moe_prepack_w4")


def moe_workspace_bytes(d: Dims) -> int:
    return int(load().moe_workspace_bytes(d))


def moe_layer_kernel_launches(d: Dims) -> int:
    return int(load().moe_layer_kernel_launches(d))


def moe_layer_projections_fused(d: Dims) -> bool:
    r = int(load().moe_layer_projections_fused(d))
    if r < 0:
        raise MoeError(-r, "moe_layer_projections_fused")
    return r == 1


def moe_stage_workspace_bytes(d: Dims) -> int:
    return int(load().moe_stage_workspace_bytes(d))


def moe_router_logits(x, router_weight, router_bias, d, logits, stream=None):
    _check(load().moe_router_logits(_p(x), _p(router_weight), _p(router_bias), d, _p(logits), _s(stream)),
           "moe_router_logits")


def moe_layer_forward_router(x, router_weight, router_bias, w_gate_up: W4, w_down: W4, d, out, logits_out,
                             topk_ids, topk_w, ws, ws_bytes, stream=None):
    _check(load().moe_layer_forward_router(_p(x), _p(router_weight), _p(router_bias), w_gate_up, w_down, d, _p(out),
                                           _p(logits_out), _p(topk_ids), _p(topk_w), _p(ws), ws_bytes, _s(stream)),
           "moe_layer_forward_router")


def moe_layer_forward_shared(x, logits, router_weight, router_bias, w_gate_up: W4, w_down: W4, shared_gate_up: W4,
                             shared_down: W4, d, out, logits_out, topk_ids, topk_w, ws, ws_bytes, stream=None):
    _check(load().moe_layer_forward_shared(_p(x), _p(logits), _p(router_weight), _p(router_bias), w_gate_up, w_down,
                                           shared_gate_up, shared_down, d, _p(out), _p(logits_out), _p(topk_ids),
                                           _p(topk_w), _p(ws), ws_bytes, _s(stream)), "moe_layer_forward_shared")


def moe_route_topk(logits, d, topk_ids, topk_w, stream=None):
    _check(load().moe_route_topk(_p(logits), d, _p(topk_ids), _p(topk_w), _s(stream)), "moe_route_topk")


def moe_permute(topk_ids, x, d, counts, offsets, sorted_token, inv_perm, x_perm, ws, ws_bytes, stream=None):
    _check(load().moe_permute(_p(topk_ids), _p(x), d, _p(counts), _p(offsets), _p(sorted_token), _p(inv_perm),
                              _p(x_perm), _p(ws), ws_bytes, _s(stream)), "moe_permute")


def moe_permute_noalloc(topk_ids, x, d, counts, offsets, sorted_token, inv_perm, x_perm, stream=None):
    _check(load().moe_permute_noalloc(_p(topk_ids), _p(x), d, _p(counts), _p(offsets), _p(sorted_token),
                                      _p(inv_perm), _p(x_perm), _s(stream)), "moe_permute_noalloc")


def moe_w4a16_gate_up_swiglu(x_perm, offsets, w_gate_up: W4, d, h, ws, ws_bytes, stream=None):
    _check(load().moe_w4a16_gate_up_swiglu(_p(x_perm), _p(offsets), w_gate_up, d, _p(h), _p(ws), ws_bytes,
                                           _s(stream)), "moe_w4a16_gate_up_swiglu")


def moe_w4a16_down(h, offsets, w_down: W4, d, y_perm, ws, ws_bytes, stream=None):
    _check(load().moe_w4a16_down(_p(h), _p(offsets), w_down, d, _p(y_perm), _p(ws), ws_bytes, _s(stream)),
           "moe_w4a16_down")


def moe_unpermute_combine(y_perm, inv_perm, topk_w, d, out, stream=None):
    _check(load().moe_unpermute_combine(_p(y_perm), _p(inv_perm), _p(topk_w), d, _p(out), _s(stream)),
           "moe_unpermute_combine")


def moe_layer_forward(x, logits, w_gate_up: W4, w_down: W4, d, out, topk_ids, topk_w, ws, ws_bytes, stream=None):
    _check(load().moe_layer_forward(_p(x), _p(logits), w_gate_up, w_down, d, _p(out), _p(topk_ids), _p(topk_w),
                                    _p(ws), ws_bytes, _s(stream)), "moe_layer_forward")


def moe_layer_forward_profiled(x, logits, w_gate_up: W4, w_down: W4, d, out, topk_ids, topk_w, ws, ws_bytes,
                               events, stream=None):
    """events: 6 torch.cuda.Event(enable_timing=True) (or None entries)."""
    arr = (ctypes.c_void_p * 6)(*[(e.cuda_event if e is not None else None) for e in events])
    _check(load().moe_layer_forward_profiled(_p(x), _p(logits), w_gate_up, w_down, d, _p(out), _p(topk_ids),
                                             _p(topk_w), _p(ws), ws_bytes, _s(stream), arr),
           "moe_layer_forward_profiled")


def moe_layer_forward_host(host_x, host_logits, w_gate_up: W4, w_down: W4, d, host_out, ws, ws_bytes, stream=None):
    _check(load().moe_layer_forward_host(_p(host_x), _p(host_logits), w_gate_up, w_down, d, _p(host_out), _p(ws),
                                         ws_bytes, _s(stream)), "moe_layer_forward_host")


def moe_host_plan_create(host_x, host_logits, w_gate_up: W4, w_down: W4, d, host_out, ws, ws_bytes, stream):
    """Returns the plan handle (an int); the caller destroys it with moe_host_plan_destroy."""
    h = ctypes.c_void_p()
    _check(load().moe_host_plan_create(_p(host_x), _p(host_logits), w_gate_up, w_down, d, _p(host_out), _p(ws),
                                       ws_bytes, _s(stream), ctypes.byref(h)), "moe_host_plan_create")
    return h.value


def moe_host_plan_run(plan):
    _check(load().moe_host_plan_run(ctypes.c_void_p(plan)), "moe_host_plan_run")


def moe_host_plan_destroy(plan):
    _check(load().moe_host_plan_destroy(ctypes.c_void_p(plan)), "moe_host_plan_destroy")


def moe_get_device_status(ws, stream=None) -> int:
    return int(load().moe_get_device_status(_p(ws), _s(stream)))


def moe_debug_dequant_table(out, stream=None):
    _check(load().moe_debug_dequant_table(_p(out), _s(stream)), "moe_debug_dequant_table")


def moe_debug_timeout_probe(ws, limit_ns: int, stream=None):
    _check(load().moe_debug_timeout_probe(_p(ws), int(limit_ns), _s(stream)), "moe_debug_timeout_probe")


def moe_debug_stream_read(src, nbytes: int, ws, stream=None):
    _check(load().moe_debug_stream_read(_p(src), int(nbytes), _p(ws), _s(stream)), "moe_debug_stream_read")


def moe_debug_counter_timeout_probe(ws, limit_ns: int, stream=None):
    _check(load().moe_debug_counter_timeout_probe(_p(ws), int(limit_ns), _s(stream)),
           "moe_debug_counter_timeout_probe")


def moe_debug_layer_forward_config(x, logits, w_gate_up: W4, w_down: W4, d, out, topk_ids, topk_w, ws, ws_bytes,
                                   token_tile: int, schedule: int, events=None, stream=None):
    """The layer with the GEMM's token-tile width and tile schedule forced (-1: the library's choice)."""
    arr = None
    if events is not None:
        arr = (ctypes.c_void_p * 6)(*[(e.cuda_event if e is not None else None) for e in events])
    _check(load().moe_debug_layer_forward_config(_p(x), _p(logits), w_gate_up, w_down, d, _p(out), _p(topk_ids),
                                                 _p(topk_w), _p(ws), ws_bytes, int(token_tile), int(schedule),
                                                 _s(stream), arr), "moe_debug_layer_forward_config")


def w4n(codes: torch.Tensor, scales: torch.Tensor, global_scale: torch.Tensor) -> W4N:
    return W4N(codes.data_ptr(), scales.data_ptr(), global_scale.data_ptr())


def moe_w4a4_workspace_bytes(d: Dims) -> int:
    return int(load().moe_w4a4_workspace_bytes(d))


def moe_w4a4_kernel_launches(d: Dims) -> int:
    return int(load().moe_w4a4_kernel_launches(d))


def moe_layer_forward_w4a4(x, logits, w_gate_up: W4N, w_down: W4N, d, out, topk_ids, topk_w, ws, ws_bytes,
                           stream=None):
    _check(load().moe_layer_forward_w4a4(_p(x), _p(logits), w_gate_up, w_down, d, _p(out), _p(topk_ids),
                                         _p(topk_w), _p(ws), ws_bytes, _s(stream)), "moe_layer_forward_w4a4")


def moe_quantize_nvfp4(x, rows_of, n: int, K: int, codes, scales, stream=None):
    _check(load().moe_quantize_nvfp4(_p(x), _p(rows_of), int(n), int(K), _p(codes), _p(scales), _s(stream)),
           "moe_quantize_nvfp4")


def moe_quantize_nvfp4_f32(x, rows_of, n: int, K: int, codes, scales, stream=None):
    _check(load().moe_quantize_nvfp4_f32(_p(x), _p(rows_of), int(n), int(K), _p(codes), _p(scales), _s(stream)),
           "moe_quantize_nvfp4_f32")


def moe_debug_w4a4_gemm(mode: int, act_codes, act_scales, offsets, w: W4N, d, out, out_scales, ws, stream=None):
    _check(load().moe_debug_w4a4_gemm(int(mode), _p(act_codes), _p(act_scales), _p(offsets), w, d, _p(out),
                                      _p(out_scales), _p(ws), _s(stream)), "moe_debug_w4a4_gemm")


def moe_layer_forward_w4a4_profiled(x, logits, w_gate_up: W4N, w_down: W4N, d, out, topk_ids, topk_w, ws, ws_bytes,
                                    events, stream=None):
    """events: 6 torch.cuda.Event(enable_timing=True) (or None entries)."""
    arr = (ctypes.c_void_p * 6)(*[(e.cuda_event if e is not None else None) for e in events])
    _check(load().moe_layer_forward_w4a4_profiled(_p(x), _p(logits), w_gate_up, w_down, d, _p(out), _p(topk_ids),
                                                  _p(topk_w), _p(ws), ws_bytes, _s(stream), arr),
           "moe_layer_forward_w4a4_profiled")
