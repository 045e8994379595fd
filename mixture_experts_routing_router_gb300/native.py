"""ctypes binding of libmoe.so: the C-ABI calls of include/moe.h under the same
names, taking torch tensors for device buffers and the current CUDA stream.

Argument marshalling only -- every step of the layer runs in the library's
CUDA kernels.  There is no fallback: if libmoe.so is missing or cannot be
loaded, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_INVALID_ROUTE = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_NONFINITE = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_CUDA = 6
MOE_ERR_UNSUPPORTED = 7
MOE_ERR_INTERNAL = 8

MOE_ACT_SWIGLU = 0
MOE_ACT_RELU2 = 1

# every symbol include/moe.h declares
EXPORTS = ("moe_workspace_size", "moe_workspace_init", "moe_route", "moe_dispatch", "moe_expert_up",
           "moe_expert_down", "moe_expert_ffn", "moe_combine", "moe_layer", "moe_status_read",
           "moe_status_string", "moe_last_error_message", "moe_dispatch_noalloc", "moe_gate",
           "moe_route_sigmoid", "moe_expert_up_fp8", "moe_expert_down_fp8", "moe_layer_fp8",
           "moe_expert_up_nvfp4", "moe_expert_down_nvfp4", "moe_layer_nvfp4", "moe_workspace_set_wait",
           "moe_timeout_site_read", "moe_ep_plan")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = last_error_message()
        super().__init__(f"{where}: status {status} ({status_string(status)})" + (f": {msg}" if msg else ""))


class moe_shape(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int32), ("hidden", ctypes.c_int32), ("experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32), ("shared", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("capacity", ctypes.c_int32), ("act", ctypes.c_int32)]


def make_shape(tokens, hidden, experts, top_k, inter, act=MOE_ACT_SWIGLU, shared=0, shared_inter=0,
               capacity=0) -> moe_shape:
    return moe_shape(tokens, hidden, experts, top_k, inter, shared, shared_inter,
                     capacity if capacity > 0 else tokens, act)


def shape_of(wl) -> moe_shape:
    """moe_shape of a synth.Workload."""
    return make_shape(wl.tokens, wl.hidden, wl.experts, wl.top_k, wl.inter, wl.act, wl.shared,
                      wl.shared_inter, wl.cap)


_lock = threading.Lock()
_lib = None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built: run mixture_experts_routing_router_gb300.build.build() "
                                   "(nvcc, sm_103a); there is no CPU fallback")
            L = ctypes.CDLL(LIB_PATH)
            P, S = ctypes.c_void_p, ctypes.c_size_t
            SP = ctypes.POINTER(moe_shape)
            sig = {
                "moe_workspace_size": [SP, ctypes.POINTER(ctypes.c_size_t)],
                "moe_workspace_init": [P, S, P],
                "moe_route": [SP, P, P, P, P, S, P],
                "moe_dispatch": [SP, P, P, P, P, P, P, P, P, S, P],
                "moe_expert_up": [SP, P, P, P, P, P, P, P, S, P],
                "moe_expert_down": [SP, P, P, P, P, P, P, P, S, P],
                "moe_expert_ffn": [SP, P, P, P, P, P, P, P, P, P, P, P, S, P],
                "moe_combine": [SP, P, P, P, P, P, P, P, S, P],
                "moe_layer": [SP, P, P, P, P, P, P, P, P, P, P, P, S, P],
                "moe_status_read": [P, P, ctypes.POINTER(ctypes.c_int)],
                "moe_dispatch_noalloc": [SP, P, P, P, P, P, P, P, P, P],
                "moe_gate": [SP, P, P, P, P, S, P],
                "moe_route_sigmoid": [SP, P, P, ctypes.c_float, P, P, P, S, P],
                "moe_expert_up_fp8": [SP, P, P, P, P, P, P, S, P],
                "moe_expert_down_fp8": [SP, P, P, P, P, P, P, S, P],
                "moe_layer_fp8": [SP, P, P, P, P, P, P, P, P, P, P, P, S, P],
                "moe_expert_up_nvfp4": [SP, P, P, P, P, P, P, P, S, P],
                "moe_expert_down_nvfp4": [SP, P, P, P, P, P, P, P, S, P],
                "moe_layer_nvfp4": [SP, P, P, P, P, P, P, P, P, P, P, P, P, P, S, P],
                "moe_workspace_set_wait": [P, S, ctypes.c_uint64, ctypes.c_int32, P],
                "moe_timeout_site_read": [P, P, ctypes.POINTER(ctypes.c_int32)],
                "moe_ep_plan": [ctypes.c_int32] * 4 + [P] * 6,
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.moe_status_string.argtypes = [ctypes.c_int]
            L.moe_status_string.restype = ctypes.c_char_p
            L.moe_last_error_message.argtypes = []
            L.moe_last_error_message.restype = ctypes.c_char_p
            _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().moe_status_string(int(status)).decode()
    except Exception:
        return "?"


def last_error_message() -> str:
    try:
        return lib().moe_last_error_message().decode()
    except Exception:
        return ""


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(st, where):
    if st != MOE_OK:
        raise MoEError(st, where)


# ---- the C-ABI calls ------------------------------------------------------
def moe_workspace_size(shape: moe_shape) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(shape), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_workspace_init")


def workspace(shape: moe_shape, device="cuda") -> torch.Tensor:
    """A zero-initialised workspace tensor of moe_workspace_size bytes."""
    return torch.zeros(moe_workspace_size(shape), dtype=torch.uint8, device=device)


def _wsb(ws):
    return ws.numel() * ws.element_size()


def moe_route(shape, logits, topk_ids, topk_w, ws, stream=None):
    _check(lib().moe_route(ctypes.byref(shape), _ptr(logits), _ptr(topk_ids), _ptr(topk_w), _ptr(ws), _wsb(ws),
                           _stream(stream)), "moe_route")


def moe_gate(shape, x, w_gate, logits, ws, stream=None):
    _check(lib().moe_gate(ctypes.byref(shape), _ptr(x), _ptr(w_gate), _ptr(logits), _ptr(ws), _wsb(ws),
                          _stream(stream)), "moe_gate")


def moe_route_sigmoid(shape, logits, bias, route_scale, topk_ids, topk_w, ws, stream=None):
    _check(lib().moe_route_sigmoid(ctypes.byref(shape), _ptr(logits), _ptr(bias), float(route_scale),
                                   _ptr(topk_ids), _ptr(topk_w), _ptr(ws), _wsb(ws), _stream(stream)),
           "moe_route_sigmoid")


def moe_dispatch(shape, x, topk_ids, counts, offsets, dest, sorted_pair, x_perm, ws, stream=None):
    _check(lib().moe_dispatch(ctypes.byref(shape), _ptr(x), _ptr(topk_ids), _ptr(counts), _ptr(offsets), _ptr(dest),
                              _ptr(sorted_pair), _ptr(x_perm), _ptr(ws), _wsb(ws), _stream(stream)), "moe_dispatch")


def moe_expert_up(shape, x_perm, offsets, w13, x, ws13, h, ws, stream=None):
    _check(lib().moe_expert_up(ctypes.byref(shape), _ptr(x_perm), _ptr(offsets), _ptr(w13), _ptr(x), _ptr(ws13),
                               _ptr(h), _ptr(ws), _wsb(ws), _stream(stream)), "moe_expert_up")


def moe_expert_down(shape, h, offsets, w2, ws2, y_perm, y_shared, ws, stream=None):
    _check(lib().moe_expert_down(ctypes.byref(shape), _ptr(h), _ptr(offsets), _ptr(w2), _ptr(ws2), _ptr(y_perm),
                                 _ptr(y_shared), _ptr(ws), _wsb(ws), _stream(stream)), "moe_expert_down")


def moe_expert_ffn(shape, x_perm, offsets, w13, w2, x, ws13, ws2, h, y_perm, y_shared, ws, stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(shape), _ptr(x_perm), _ptr(offsets), _ptr(w13), _ptr(w2), _ptr(x),
                                _ptr(ws13), _ptr(ws2), _ptr(h), _ptr(y_perm), _ptr(y_shared), _ptr(ws), _wsb(ws),
                                _stream(stream)), "moe_expert_ffn")


def moe_combine(shape, y_perm, dest, topk_w, y_shared, out, ws, stream=None, residual=None):
    _check(lib().moe_combine(ctypes.byref(shape), _ptr(y_perm), _ptr(dest), _ptr(topk_w), _ptr(y_shared),
                             _ptr(residual), _ptr(out), _ptr(ws), _wsb(ws), _stream(stream)), "moe_combine")


def moe_layer(shape, logits, ids_in, w_in, x, w13, w2, ws13, ws2, out, ws, stream=None, residual=None):
    _check(lib().moe_layer(ctypes.byref(shape), _ptr(logits), _ptr(ids_in), _ptr(w_in), _ptr(x), _ptr(w13),
                           _ptr(w2), _ptr(ws13), _ptr(ws2), _ptr(residual), _ptr(out), _ptr(ws), _wsb(ws),
                           _stream(stream)), "moe_layer")


def moe_expert_up_fp8(shape, x_perm, offsets, w13, w13_scale, h, ws, stream=None):
    """Up projection with FP8 E4M3 weights (uint8 [E, up, H]) and FP32 row scales ([E, up])."""
    _check(lib().moe_expert_up_fp8(ctypes.byref(shape), _ptr(x_perm), _ptr(offsets), _ptr(w13), _ptr(w13_scale),
                                   _ptr(h), _ptr(ws), _wsb(ws), _stream(stream)), "moe_expert_up_fp8")


def moe_expert_down_fp8(shape, h, offsets, w2, w2_scale, y_perm, ws, stream=None):
    """Down projection with FP8 E4M3 weights (uint8 [E, H, I]) and FP32 row scales ([E, H])."""
    _check(lib().moe_expert_down_fp8(ctypes.byref(shape), _ptr(h), _ptr(offsets), _ptr(w2), _ptr(w2_scale),
                                     _ptr(y_perm), _ptr(ws), _wsb(ws), _stream(stream)), "moe_expert_down_fp8")


def moe_layer_fp8(shape, logits, ids_in, w_in, x, w13, w13_scale, w2, w2_scale, out, ws, stream=None,
                  residual=None):
    """The layer with FP8 E4M3 expert weights (no shared experts)."""
    _check(lib().moe_layer_fp8(ctypes.byref(shape), _ptr(logits), _ptr(ids_in), _ptr(w_in), _ptr(x), _ptr(w13),
                               _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(residual), _ptr(out), _ptr(ws),
                               _wsb(ws), _stream(stream)), "moe_layer_fp8")


def moe_expert_up_nvfp4(shape, x_perm, offsets, w13, w13_bscale, w13_scale, h, ws, stream=None):
    """Up projection with NVFP4 weights: codes uint8 [E, up, H/2], E4M3 block
    scales uint8 [E, up, 16*ceil(H/256)], FP32 row scales [E, up]."""
    _check(lib().moe_expert_up_nvfp4(ctypes.byref(shape), _ptr(x_perm), _ptr(offsets), _ptr(w13), _ptr(w13_bscale),
                                     _ptr(w13_scale), _ptr(h), _ptr(ws), _wsb(ws), _stream(stream)),
           "moe_expert_up_nvfp4")


def moe_expert_down_nvfp4(shape, h, offsets, w2, w2_bscale, w2_scale, y_perm, ws, stream=None):
    """Down projection with NVFP4 weights: codes uint8 [E, H, I/2], block
    scales uint8 [E, H, 16*ceil(I/256)], FP32 row scales [E, H]."""
    _check(lib().moe_expert_down_nvfp4(ctypes.byref(shape), _ptr(h), _ptr(offsets), _ptr(w2), _ptr(w2_bscale),
                                       _ptr(w2_scale), _ptr(y_perm), _ptr(ws), _wsb(ws), _stream(stream)),
           "moe_expert_down_nvfp4")


def moe_layer_nvfp4(shape, logits, ids_in, w_in, x, w13, w13_bscale, w13_scale, w2, w2_bscale, w2_scale, out, ws,
                    stream=None, residual=None):
    """The layer with NVFP4 expert weights (no shared experts)."""
    _check(lib().moe_layer_nvfp4(ctypes.byref(shape), _ptr(logits), _ptr(ids_in), _ptr(w_in), _ptr(x), _ptr(w13),
                                 _ptr(w13_bscale), _ptr(w13_scale), _ptr(w2), _ptr(w2_bscale), _ptr(w2_scale),
                                 _ptr(residual), _ptr(out), _ptr(ws), _wsb(ws), _stream(stream)), "moe_layer_nvfp4")


def moe_dispatch_noalloc(shape, x, topk_ids, counts, offsets, dest, sorted_pair, x_perm, device_status=None,
                         stream=None):
    """moe_dispatch without a workspace (static scratch inside the library)."""
    _check(lib().moe_dispatch_noalloc(ctypes.byref(shape), _ptr(x), _ptr(topk_ids), _ptr(counts), _ptr(offsets),
                                      _ptr(dest), _ptr(sorted_pair), _ptr(x_perm), _ptr(device_status),
                                      _stream(stream)), "moe_dispatch_noalloc")


def moe_status_read(ws, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(lib().moe_status_read(_ptr(ws), _stream(stream), ctypes.byref(st)), "moe_status_read")
    return st.value


def moe_workspace_set_wait(ws, lookback_wait_ns: int, count_tile_skip: int = 0, stream=None):
    """Test controls of the count kernel's bounded look-back wait."""
    _check(lib().moe_workspace_set_wait(_ptr(ws), _wsb(ws), int(lookback_wait_ns), int(count_tile_skip),
                                        _stream(stream)), "moe_workspace_set_wait")


def moe_timeout_site_read(ws, stream=None) -> int:
    site = ctypes.c_int32(0)
    _check(lib().moe_timeout_site_read(_ptr(ws), _stream(stream), ctypes.byref(site)), "moe_timeout_site_read")
    return site.value


def moe_ep_plan(experts: int, world: int, rank: int, capacity: int, counts_all):
    """Host-side plan of the expert-parallel exchange (numpy in, numpy out):
    -> (status, dict(send_offsets [E+1], recv_offsets [el+1], recv_slot [world, el],
    peer_send [world], peer_recv [world])).  The status is MOE_OK or
    MOE_ERR_CAPACITY (the plan is written either way); other errors raise."""
    import numpy as np
    ca = np.ascontiguousarray(counts_all, dtype=np.int32)
    if ca.shape != (world, experts):
        raise ValueError(f"counts_all must be [{world}, {experts}], got {ca.shape}")
    e0, e1 = rank * experts // world, (rank + 1) * experts // world
    out = dict(send_offsets=np.zeros(experts + 1, np.int32), recv_offsets=np.zeros(e1 - e0 + 1, np.int32),
               recv_slot=np.zeros((world, e1 - e0), np.int32), peer_send=np.zeros(world, np.int32),
               peer_recv=np.zeros(world, np.int32))
    p = lambda a: ctypes.c_void_p(a.ctypes.data)
    st = lib().moe_ep_plan(experts, world, rank, capacity, p(ca), p(out["send_offsets"]), p(out["recv_offsets"]),
                           p(out["recv_slot"]), p(out["peer_send"]), p(out["peer_recv"]))
    if st not in (MOE_OK, MOE_ERR_CAPACITY):
        raise MoEError(st, "moe_ep_plan")
    return st, out
