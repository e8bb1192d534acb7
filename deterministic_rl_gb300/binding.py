"""ctypes binding of libmoedet (include/moe_det.h): argument marshalling only.

Every step of the layer runs in the CUDA library; this module converts torch
tensors into device pointers and the dims/weights structs, and nothing else.
There is no fallback: if libmoedet.so is missing or cannot be loaded, loading
raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoedet.so")

MOE_OK = 0
MOE_ERR_ARG = 1
MOE_ERR_SHAPE = 2
MOE_ERR_ALIGN = 3
MOE_ERR_WORKSPACE = 4
MOE_ERR_BAD_IDS = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_CUDA = 7
MOE_ERR_UNSUPPORTED = 8

MOE_W_BF16 = 0
MOE_W_MXFP8 = 1
MOE_W_NVFP4 = 2
MOE_W_MXFP8_ACT = 3

# Every function the header declares, in declaration order.
EXPORTED = ("moe_workspace_size", "moe_workspace_layout", "moe_route", "moe_forward",
            "moe_forward_replay", "moe_get_status", "moe_status_str", "moe_set_stage_events",
            "moe_route_static", "moe_forward_replay_filtered", "moe_backward_weights_size",
            "moe_backward_prepare_weights", "moe_backward_workspace_size",
            "moe_backward_workspace_layout", "moe_set_backward_stage_events", "moe_backward",
            "moe_forward_train", "moe_backward_saved", "moe_packed_weights_size",
            "moe_pack_weights")

STAGES = ("router_gemm", "topk", "dispatch", "gather", "gate_up", "down", "combine")
BWD_STAGES = ("prepare", "route", "dispatch", "gate_up", "down", "gate", "dy", "dh", "swiglu",
              "dxp", "dx", "transpose", "wgrad_down", "wgrad_gate_up")


class moe_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("F", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("wfmt", ctypes.c_int32), ("out_fp32", ctypes.c_int32)]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "router_bias", "w_gate", "w_up", "w_down", "s_gate", "s_up",
                 "s_down", "ws_gate", "ws_up", "ws_down", "gs_gate", "gs_up", "gs_down",
                 "w_gate_up")]


class moe_ws_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "logits", "valid", "cnt", "off", "perm", "inv", "xp", "h", "y",
                 "ysh", "xq", "sx", "sxp", "sh", "hq", "total")]


class moe_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("d_router", "d_gate", "d_up", "d_down", "ds_gate", "ds_up", "ds_down")]


class moe_bwd_ws_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "logits", "valid", "cnt", "off", "perm", "inv", "xp", "h", "y",
                 "ids", "gates", "poff", "a", "b", "dg", "dl", "dyq", "dh", "dabq", "dxp",
                 "xpt", "dyt", "ht", "dabt", "kpad", "total")]


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_str(code)}")


_lib = None


def load(path: str = LIB_PATH):
    """Load libmoedet.so (built by deterministic_rl_gb300.build) and declare
    the signatures.  Raises OSError when the library is not there."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} not found: build it with deterministic_rl_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    D = ctypes.POINTER(moe_dims)
    W = ctypes.POINTER(moe_weights)
    lib.moe_workspace_size.restype = ctypes.c_size_t
    lib.moe_workspace_size.argtypes = [D]
    lib.moe_workspace_layout.restype = ctypes.c_int
    lib.moe_workspace_layout.argtypes = [D, ctypes.POINTER(moe_ws_layout)]
    lib.moe_route.restype = ctypes.c_int
    lib.moe_route.argtypes = [D, P, W, P, P, P, ctypes.c_size_t, P]
    lib.moe_forward.restype = ctypes.c_int
    lib.moe_forward.argtypes = [D, P, W, P, P, P, P, ctypes.c_size_t, P]
    lib.moe_forward_replay.restype = ctypes.c_int
    lib.moe_forward_replay.argtypes = [D, P, W, P, P, P, P, P, ctypes.c_size_t, P]
    lib.moe_get_status.restype = ctypes.c_int
    lib.moe_get_status.argtypes = [P, P]
    lib.moe_status_str.restype = ctypes.c_char_p
    lib.moe_status_str.argtypes = [ctypes.c_int]
    lib.moe_set_stage_events.restype = ctypes.c_int
    lib.moe_set_stage_events.argtypes = [ctypes.c_void_p]
    lib.moe_forward_replay_filtered.restype = ctypes.c_int
    lib.moe_forward_replay_filtered.argtypes = [D, P, W, P, ctypes.c_float, P, P, P, P,
                                                ctypes.c_size_t, P]
    lib.moe_route_static.restype = ctypes.c_int
    lib.moe_route_static.argtypes = [D, P, W, P, P, P]
    lib.moe_backward_weights_size.restype = ctypes.c_size_t
    lib.moe_backward_weights_size.argtypes = [D]
    lib.moe_backward_prepare_weights.restype = ctypes.c_int
    lib.moe_backward_prepare_weights.argtypes = [D, W, P, ctypes.c_size_t, P]
    lib.moe_backward_workspace_size.restype = ctypes.c_size_t
    lib.moe_backward_workspace_size.argtypes = [D]
    lib.moe_backward_workspace_layout.restype = ctypes.c_int
    lib.moe_backward_workspace_layout.argtypes = [D, ctypes.POINTER(moe_bwd_ws_layout)]
    lib.moe_packed_weights_size.restype = ctypes.c_size_t
    lib.moe_packed_weights_size.argtypes = [D]
    lib.moe_pack_weights.restype = ctypes.c_int
    lib.moe_pack_weights.argtypes = [D, W, P, ctypes.c_size_t, P]
    lib.moe_forward_train.restype = ctypes.c_int
    lib.moe_forward_train.argtypes = [D, P, W, P, P, P, P, P, ctypes.c_size_t, P]
    lib.moe_backward_saved.restype = ctypes.c_int
    lib.moe_backward_saved.argtypes = [D, W, P, P, P, ctypes.POINTER(moe_grads), P,
                                       ctypes.c_size_t, P]
    lib.moe_set_backward_stage_events.restype = ctypes.c_int
    lib.moe_set_backward_stage_events.argtypes = [ctypes.c_void_p]
    lib.moe_backward.restype = ctypes.c_int
    lib.moe_backward.argtypes = [D, P, W, P, P, P, P, ctypes.POINTER(moe_grads), P,
                                 ctypes.c_size_t, P]
    _lib = lib
    return lib


def status_str(code: int) -> str:
    return load().moe_status_str(int(code)).decode()


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class Dims:
    T: int
    d: int
    E: int
    k: int
    F: int
    n_shared: int
    wfmt: int = MOE_W_BF16
    out_fp32: int = 0

    def c(self) -> moe_dims:
        return moe_dims(self.T, self.d, self.E, self.k, self.F, self.n_shared, self.wfmt,
                        self.out_fp32)


def make_weights(w_router, router_bias, w_gate, w_up, w_down, s_gate=None, s_up=None,
                 s_down=None, ws_gate=None, ws_up=None, ws_down=None, gs_gate=None, gs_up=None,
                 gs_down=None, w_gate_up=None) -> moe_weights:
    return moe_weights(*(_p(t) for t in (w_router, router_bias, w_gate, w_up, w_down, s_gate,
                                         s_up, s_down, ws_gate, ws_up, ws_down, gs_gate, gs_up,
                                         gs_down, w_gate_up)))


def moe_workspace_size(dims: Dims) -> int:
    return int(load().moe_workspace_size(ctypes.byref(dims.c())))


def moe_workspace_layout(dims: Dims) -> moe_ws_layout:
    out = moe_ws_layout()
    rc = load().moe_workspace_layout(ctypes.byref(dims.c()), ctypes.byref(out))
    if rc != MOE_OK:
        raise MoEError(rc, "moe_workspace_layout")
    return out


def moe_route(dims: Dims, x, weights: moe_weights, ids_out, gates_out, ws,
              stream=None, check: bool = True) -> int:
    rc = load().moe_route(ctypes.byref(dims.c()), _p(x), ctypes.byref(weights), _p(ids_out),
                          _p(gates_out), _p(ws), ws.numel() * ws.element_size(), _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_route")
    return rc


def moe_forward(dims: Dims, x, weights: moe_weights, out, ids_out, gates_out, ws,
                stream=None, check: bool = True) -> int:
    rc = load().moe_forward(ctypes.byref(dims.c()), _p(x), ctypes.byref(weights), _p(out),
                            _p(ids_out), _p(gates_out), _p(ws), ws.numel() * ws.element_size(),
                            _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_forward")
    return rc


def moe_forward_replay(dims: Dims, x, weights: moe_weights, ids_in, out, ids_out, gates_out,
                       ws, stream=None, check: bool = True) -> int:
    rc = load().moe_forward_replay(ctypes.byref(dims.c()), _p(x), ctypes.byref(weights),
                                   _p(ids_in), _p(out), _p(ids_out), _p(gates_out), _p(ws),
                                   ws.numel() * ws.element_size(), _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_forward_replay")
    return rc


def moe_get_status(ws, stream=None) -> int:
    return int(load().moe_get_status(_p(ws), _stream(stream)))


def moe_status_str(code: int) -> str:
    return status_str(code)


def moe_set_stage_events(events) -> int:
    """events: None, or a sequence of 2 * len(STAGES) torch.cuda.Event objects
    (created with enable_timing=True and already recorded once so that their
    handles exist).  See the header for the semantics."""
    if events is None:
        return int(load().moe_set_stage_events(None))
    assert len(events) == 2 * len(STAGES)
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return int(load().moe_set_stage_events(ctypes.cast(arr, ctypes.c_void_p)))


def moe_route_static(dims: Dims, x, weights: moe_weights, ids_out, gates_out, stream=None,
                     check: bool = True) -> int:
    """Routing whose scratch is the library's static device array: for callers
    that cannot allocate device memory (see the header)."""
    rc = load().moe_route_static(ctypes.byref(dims.c()), _p(x), ctypes.byref(weights),
                                 _p(ids_out), _p(gates_out), _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_route_static")
    return rc


def moe_forward_replay_filtered(dims: Dims, x, weights: moe_weights, ids_in, tau: float, out,
                                ids_out, gates_out, ws, stream=None, check: bool = True) -> int:
    rc = load().moe_forward_replay_filtered(ctypes.byref(dims.c()), _p(x), ctypes.byref(weights),
                                            _p(ids_in), float(tau), _p(out), _p(ids_out),
                                            _p(gates_out), _p(ws), ws.numel() * ws.element_size(),
                                            _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_forward_replay_filtered")
    return rc


# ---- backward ----

def make_grads(d_router, d_gate, d_up, d_down, ds_gate=None, ds_up=None,
               ds_down=None) -> moe_grads:
    return moe_grads(*(_p(t) for t in (d_router, d_gate, d_up, d_down, ds_gate, ds_up, ds_down)))


def moe_backward_weights_size(dims: Dims) -> int:
    return int(load().moe_backward_weights_size(ctypes.byref(dims.c())))


def moe_backward_prepare_weights(dims: Dims, weights: moe_weights, wt, stream=None,
                                 check: bool = True) -> int:
    rc = load().moe_backward_prepare_weights(ctypes.byref(dims.c()), ctypes.byref(weights),
                                             _p(wt), wt.numel() * wt.element_size(),
                                             _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_backward_prepare_weights")
    return rc


def moe_backward_workspace_size(dims: Dims) -> int:
    return int(load().moe_backward_workspace_size(ctypes.byref(dims.c())))


def moe_backward_workspace_layout(dims: Dims) -> moe_bwd_ws_layout:
    out = moe_bwd_ws_layout()
    rc = load().moe_backward_workspace_layout(ctypes.byref(dims.c()), ctypes.byref(out))
    if rc != MOE_OK:
        raise MoEError(rc, "moe_backward_workspace_layout")
    return out


def moe_backward(dims: Dims, x, weights: moe_weights, wt, ids, dout, dx, grads: moe_grads, ws,
                 stream=None, check: bool = True) -> int:
    rc = load().moe_backward(ctypes.byref(dims.c()), _p(x), ctypes.byref(weights), _p(wt),
                             _p(ids), _p(dout), _p(dx), ctypes.byref(grads), _p(ws),
                             ws.numel() * ws.element_size(), _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_backward")
    return rc


def moe_set_backward_stage_events(events) -> int:
    """events: None, or 2 * len(BWD_STAGES) recorded torch.cuda.Event objects."""
    if events is None:
        return int(load().moe_set_backward_stage_events(None))
    assert len(events) == 2 * len(BWD_STAGES)
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return int(load().moe_set_backward_stage_events(ctypes.cast(arr, ctypes.c_void_p)))


def moe_forward_train(dims: Dims, x, weights: moe_weights, ids_in, out, ids_out, gates_out, ws,
                      stream=None, check: bool = True) -> int:
    rc = load().moe_forward_train(ctypes.byref(dims.c()), _p(x), ctypes.byref(weights),
                                  _p(ids_in), _p(out), _p(ids_out), _p(gates_out), _p(ws),
                                  ws.numel() * ws.element_size(), _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_forward_train")
    return rc


def moe_backward_saved(dims: Dims, weights: moe_weights, wt, dout, dx, grads: moe_grads, ws,
                       stream=None, check: bool = True) -> int:
    rc = load().moe_backward_saved(ctypes.byref(dims.c()), ctypes.byref(weights), _p(wt),
                                   _p(dout), _p(dx), ctypes.byref(grads), _p(ws),
                                   ws.numel() * ws.element_size(), _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_backward_saved")
    return rc


def moe_packed_weights_size(dims: Dims) -> int:
    return int(load().moe_packed_weights_size(ctypes.byref(dims.c())))


def moe_pack_weights(dims: Dims, weights: moe_weights, packed, stream=None,
                     check: bool = True) -> int:
    rc = load().moe_pack_weights(ctypes.byref(dims.c()), ctypes.byref(weights), _p(packed),
                                 packed.numel() * packed.element_size(), _stream(stream))
    if check and rc != MOE_OK:
        raise MoEError(rc, "moe_pack_weights")
    return rc

