"""Thin ctypes binding of libmoe_gb300.so (declared in include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions keep the C names; tensors are torch tensors (device memory)
or raw integer device addresses.  A non-OK status raises MoeError carrying the
status and the library's message.  Importing this module fails loudly when the
library has not been built -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK, MOE_EINVAL, MOE_EDIMS, MOE_ESCALE, MOE_ENOMEM, MOE_ECUDA, MOE_EWORKSPACE, MOE_EDEVICE = range(8)
STATUS_NAMES = ["MOE_OK", "MOE_EINVAL", "MOE_EDIMS", "MOE_ESCALE", "MOE_ENOMEM", "MOE_ECUDA", "MOE_EWORKSPACE",
                "MOE_EDEVICE"]
MOE_W_MXFP4, MOE_W_BF16, MOE_W_INT4G32 = 0, 1, 2

# every symbol include/moe.h declares
EXPORTED = ("moe_load_weights", "moe_workspace_bytes", "moe_forward", "moe_forward_routed", "moe_set_expert_range",
            "moe_route_sigmoid", "moe_dense_sliced_forward", "moe_sync_status", "moe_profile_enable",
            "moe_profile_read", "moe_route_static", "moe_route_static_status", "moe_graph_create",
            "moe_graph_launch", "moe_graph_free", "moe_debug_expire_next_wait", "moe_last_error", "moe_free")
STAGES = ("routing", "grouping", "gate_up", "down", "combine", "layer")


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES[status] if 0 <= status < 8 else status}: {message}")
        self.status = status


class MoeConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("n_shared", ctypes.c_int), ("k_max", ctypes.c_int), ("n_slices", ctypes.c_int),
                ("fmt", ctypes.c_int)]


class MoeMx(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zeros", ctypes.c_void_p)]


class MoeHostIO(ctypes.Structure):
    _fields_ = [("x_host", ctypes.c_void_p), ("logits_host", ctypes.c_void_p), ("ids_host", ctypes.c_void_p),
                ("w_host", ctypes.c_void_p), ("out_host", ctypes.c_void_p)]


class MoeRoutingOut(ctypes.Structure):
    _fields_ = [("topk_ids", ctypes.c_void_p), ("topk_w", ctypes.c_void_p), ("expert_offsets", ctypes.c_void_p),
                ("sorted_slot", ctypes.c_void_p), ("slot_pos", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m mxfp4_routed_expert_router_gb300.build`"
                          " (or __graft_entry__.build())")
    L = ctypes.CDLL(LIB_PATH)
    vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.moe_load_weights.argtypes = [ctypes.POINTER(MoeConfig), ctypes.POINTER(MoeMx), ctypes.POINTER(MoeMx), vp,
                                   ctypes.POINTER(vp)]
    L.moe_load_weights.restype = ci
    L.moe_workspace_bytes.argtypes = [vp, ci, ci]
    L.moe_workspace_bytes.restype = sz
    L.moe_forward.argtypes = [vp, vp, vp, ci, ci, vp, ci, vp, sz, ctypes.POINTER(MoeRoutingOut), vp]
    L.moe_forward.restype = ci
    L.moe_forward_routed.argtypes = [vp, vp, vp, vp, ci, ci, vp, ci, vp, sz, ctypes.POINTER(MoeRoutingOut), vp]
    L.moe_forward_routed.restype = ci
    L.moe_set_expert_range.argtypes = [vp, ci, ci]
    L.moe_set_expert_range.restype = ci
    L.moe_route_sigmoid.argtypes = [vp, vp, ci, ci, ci, ctypes.c_float, vp, vp, vp]
    L.moe_route_sigmoid.restype = ci
    L.moe_graph_create.argtypes = [vp, vp, vp, vp, vp, ci, ci, vp, ci, vp, sz, ctypes.POINTER(MoeHostIO),
                                   ctypes.POINTER(vp)]
    L.moe_graph_create.restype = ci
    L.moe_graph_launch.argtypes = [vp, vp]
    L.moe_graph_launch.restype = ci
    L.moe_graph_free.argtypes = [vp]
    L.moe_graph_free.restype = None
    L.moe_dense_sliced_forward.argtypes = [vp, vp, ci, vp, ci, vp, sz, vp]
    L.moe_dense_sliced_forward.restype = ci
    L.moe_sync_status.argtypes = [vp, vp]
    L.moe_sync_status.restype = ci
    L.moe_profile_enable.argtypes = [vp, ci]
    L.moe_profile_enable.restype = ci
    L.moe_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ci]
    L.moe_profile_read.restype = ci
    L.moe_route_static.argtypes = [vp, ci, ci, ci, vp, vp, vp, vp, vp, vp]
    L.moe_route_static.restype = ci
    L.moe_route_static_status.argtypes = [vp]
    L.moe_route_static_status.restype = ci
    L.moe_debug_expire_next_wait.argtypes = [vp, ci]
    L.moe_debug_expire_next_wait.restype = ci
    L.moe_last_error.argtypes = []
    L.moe_last_error.restype = ctypes.c_char_p
    L.moe_free.argtypes = [vp]
    L.moe_free.restype = None
    return L


lib = _load()


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, moe_last_error())


def moe_last_error() -> str:
    return lib.moe_last_error().decode()


def moe_load_weights(cfg: MoeConfig, gate_up: Sequence[Tuple], down: Sequence[Tuple], stream=None) -> int:
    """Copy weights into the library; gate_up / down are sequences of
    (codes, scales_or_None) or, for INT4G32, (codes, scales, zeros_or_None)."""
    def mx(m):
        return MoeMx(_ptr(m[0]), _ptr(m[1]), _ptr(m[2]) if len(m) > 2 else None)

    gu = (MoeMx * max(1, len(gate_up)))(*[mx(m) for m in gate_up])
    dn = (MoeMx * max(1, len(down)))(*[mx(m) for m in down])
    h = ctypes.c_void_p()
    _check(lib.moe_load_weights(ctypes.byref(cfg), gu, dn, _stream(stream), ctypes.byref(h)))
    return h.value


def moe_workspace_bytes(handle: int, T: int, k: int) -> int:
    return int(lib.moe_workspace_bytes(handle, T, k))


def moe_forward(handle: int, x_bf16, router_logits, T: int, k: int, out_fp32, accumulate: bool, workspace,
                ws_bytes: int, routing: Optional[MoeRoutingOut] = None, stream=None) -> None:
    _check(lib.moe_forward(handle, _ptr(x_bf16), _ptr(router_logits), T, k, _ptr(out_fp32), int(bool(accumulate)),
                           _ptr(workspace), ws_bytes, ctypes.byref(routing) if routing is not None else None,
                           _stream(stream)))


def moe_forward_routed(handle: int, x_bf16, topk_ids, topk_w, T: int, k: int, out_fp32, accumulate: bool, workspace,
                       ws_bytes: int, routing: Optional[MoeRoutingOut] = None, stream=None) -> None:
    _check(lib.moe_forward_routed(handle, _ptr(x_bf16), _ptr(topk_ids), _ptr(topk_w), T, k, _ptr(out_fp32),
                                  int(bool(accumulate)), _ptr(workspace), ws_bytes,
                                  ctypes.byref(routing) if routing is not None else None, _stream(stream)))


def moe_set_expert_range(handle: int, expert_base: int, n_experts_total: int) -> None:
    _check(lib.moe_set_expert_range(handle, int(expert_base), int(n_experts_total)))


def moe_route_sigmoid(router_logits, bias, T: int, E: int, k: int, routed_scale: float, topk_ids, topk_w,
                      stream=None) -> None:
    _check(lib.moe_route_sigmoid(_ptr(router_logits), _ptr(bias), T, E, k, float(routed_scale), _ptr(topk_ids),
                                 _ptr(topk_w), _stream(stream)))


def moe_graph_create(handle: int, x_bf16, router_logits, topk_ids, topk_w, T: int, k: int, out_fp32,
                     accumulate: bool, workspace, ws_bytes: int, x_host=None, logits_host=None, ids_host=None,
                     w_host=None, out_host=None) -> int:
    """Capture one forward call into a CUDA graph; the *_host buffers (pinned host memory, optional) add the
    step's input and output copies to the graph."""
    io = MoeHostIO(_ptr(x_host), _ptr(logits_host), _ptr(ids_host), _ptr(w_host), _ptr(out_host))
    any_io = any(v is not None for v in (x_host, logits_host, ids_host, w_host, out_host))
    g = ctypes.c_void_p()
    _check(lib.moe_graph_create(handle, _ptr(x_bf16), _ptr(router_logits), _ptr(topk_ids), _ptr(topk_w), T, k,
                                _ptr(out_fp32), int(bool(accumulate)), _ptr(workspace), ws_bytes,
                                ctypes.byref(io) if any_io else None, ctypes.byref(g)))
    return g.value


def moe_graph_launch(graph: int, stream=None) -> None:
    _check(lib.moe_graph_launch(graph, _stream(stream)))


def moe_graph_free(graph: int) -> None:
    lib.moe_graph_free(graph)


def moe_dense_sliced_forward(handle: int, x_bf16, T: int, out_fp32, accumulate: bool, workspace, ws_bytes: int,
                             stream=None) -> None:
    _check(lib.moe_dense_sliced_forward(handle, _ptr(x_bf16), T, _ptr(out_fp32), int(bool(accumulate)),
                                        _ptr(workspace), ws_bytes, _stream(stream)))


def moe_sync_status(handle: int, stream=None) -> None:
    _check(lib.moe_sync_status(handle, _stream(stream)))


def moe_profile_enable(handle: int, enable: bool = True) -> None:
    _check(lib.moe_profile_enable(handle, int(bool(enable))))


def moe_profile_read(handle: int) -> dict:
    """Stage durations (ms) of the most recent profiled forward call."""
    buf = (ctypes.c_float * len(STAGES))()
    n = lib.moe_profile_read(handle, buf, len(STAGES))
    if n < 0:
        raise MoeError(MOE_EINVAL, "no profiled call")
    return {STAGES[i]: float(buf[i]) for i in range(n)}


def moe_route_static(router_logits, T: int, E: int, k: int, topk_ids, topk_w, expert_offsets, sorted_slot,
                     slot_pos, stream=None) -> None:
    """Routing and grouping with the library's fixed scratch; allocates nothing (see include/moe.h)."""
    _check(lib.moe_route_static(_ptr(router_logits), T, E, k, _ptr(topk_ids), _ptr(topk_w), _ptr(expert_offsets),
                                _ptr(sorted_slot), _ptr(slot_pos), _stream(stream)))


def moe_route_static_status(stream=None) -> None:
    """Raise MoeError(MOE_EDEVICE) if the most recent moe_route_static call on this device flagged a device error."""
    _check(lib.moe_route_static_status(_stream(stream)))


def moe_debug_expire_next_wait(handle: int, limit_us: int) -> None:
    """Test hook: the next single-kernel launch on this handle lets its completion wait expire (include/moe.h)."""
    _check(lib.moe_debug_expire_next_wait(handle, int(limit_us)))


def moe_free(handle: int) -> None:
    lib.moe_free(handle)


def routing_out(topk_ids=None, topk_w=None, expert_offsets=None, sorted_slot=None, slot_pos=None) -> MoeRoutingOut:
    return MoeRoutingOut(_ptr(topk_ids), _ptr(topk_w), _ptr(expert_offsets), _ptr(sorted_slot), _ptr(slot_pos))
