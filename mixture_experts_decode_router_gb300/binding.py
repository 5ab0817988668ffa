"""ctypes binding of libmoe_gb300.so (the C ABI of ``include/moe.h``).

Argument marshalling only: the functions here have the C names, turn tensors
into device pointers and a torch stream into a ``cudaStream_t``, and return the
C status.  Every step of the layer runs in the library's CUDA kernels; if the
library cannot be loaded the import fails loudly -- there is no other path.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

# ---------------------------------------------------------------- C types

MOE_OK = 0
MOE_ERR_NULL = 1
MOE_ERR_INVALID_CONFIG = 2
MOE_ERR_UNSUPPORTED = 3
MOE_ERR_WORKSPACE = 4
MOE_ERR_CUDA = 5
MOE_ERR_ALIGNMENT = 6
MOE_ERR_ALIAS = 7
MOE_ERR_HOST_MEMORY = 8

MOE_ROUTE_SOFTMAX = 0
MOE_ROUTE_SIGMOID_BIAS = 1
MOE_W_BF16 = 0
MOE_W_FP8_B128 = 1
MOE_W_NVFP4 = 2
MOE_PATH_AUTO = 0
MOE_PATH_TOKEN_MAJOR = 1
MOE_PATH_GROUPED = 2

# Every function include/moe.h declares.
EXPORTED = ("moe_workspace_bytes", "moe_route", "moe_experts", "moe_forward",
            "moe_forward_timed", "moe_forward_static_ws", "moe_static_workspace_check",
            "moe_workspace_check", "moe_status_string", "moe_abi_version")

MOE_STATIC_WORKSPACE_BYTES = 16 << 20


class moe_config_t(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("routing", ctypes.c_int32),
                ("norm_topk_prob", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("expert_fmt", ctypes.c_int32), ("path", ctypes.c_int32),
                ("rms_norm_eps", ctypes.c_float), ("expert_begin", ctypes.c_int32),
                ("expert_end", ctypes.c_int32), ("exclude_shared", ctypes.c_int32),
                ("accumulate", ctypes.c_int32), ("router_fmt", ctypes.c_int32)]


class moe_qmat_t(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("scale2", ctypes.c_void_p)]


class moe_weights_t(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("correction_bias", ctypes.c_void_p),
                ("gate", moe_qmat_t), ("up", moe_qmat_t), ("down", moe_qmat_t),
                ("sh_gate", moe_qmat_t), ("sh_up", moe_qmat_t), ("sh_down", moe_qmat_t),
                ("shared_gate_w", ctypes.c_void_p), ("pre_expert_norm_w", ctypes.c_void_p),
                ("router_q", moe_qmat_t)]


_lib: Optional[ctypes.CDLL] = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) libmoe_gb300.so; raises if impossible."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and _build._stale():
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe_gb300.so is missing at {path}: run "
                           "`python -m mixture_experts_decode_router_gb300.build`")
    lib = ctypes.CDLL(path)
    P, S, I32, F = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_float
    cfgp, wp = ctypes.POINTER(moe_config_t), ctypes.POINTER(moe_weights_t)
    lib.moe_workspace_bytes.argtypes = [cfgp, I32]
    lib.moe_workspace_bytes.restype = S
    lib.moe_route.argtypes = [cfgp, wp, P, I32, P, P, P, P, S, P]
    lib.moe_route.restype = ctypes.c_int
    lib.moe_experts.argtypes = [cfgp, wp, P, I32, P, P, P, P, S, P]
    lib.moe_experts.restype = ctypes.c_int
    lib.moe_forward.argtypes = [cfgp, wp, P, I32, P, P, P, P, S, P]
    lib.moe_forward.restype = ctypes.c_int
    lib.moe_forward_timed.argtypes = [cfgp, wp, P, I32, P, P, P, P, S, P, P, I32,
                                      ctypes.POINTER(I32)]
    lib.moe_forward_timed.restype = ctypes.c_int
    lib.moe_forward_static_ws.argtypes = [cfgp, wp, P, I32, P, P, P, P]
    lib.moe_forward_static_ws.restype = ctypes.c_int
    lib.moe_static_workspace_check.argtypes = [ctypes.POINTER(I32), ctypes.POINTER(P), P]
    lib.moe_static_workspace_check.restype = ctypes.c_int
    lib.moe_workspace_check.argtypes = [P, S, ctypes.POINTER(I32), P]
    lib.moe_workspace_check.restype = ctypes.c_int
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_abi_version.argtypes = []
    lib.moe_abi_version.restype = I32
    _lib = lib
    return lib


# ---------------------------------------------------------------- marshalling

def _ptr(t) -> Optional[int]:
    """A tensor's device pointer, an int pointer as is, None -> NULL."""
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


def _ref(obj):
    """ctypes.byref, or a NULL pointer for None."""
    return None if obj is None else ctypes.byref(obj)


def moe_workspace_bytes(cfg: moe_config_t, max_tokens: int) -> int:
    return load().moe_workspace_bytes(_ref(cfg), int(max_tokens))


def moe_route(cfg, wts, x, n, idx, w, logits, ws, ws_bytes, stream=None) -> int:
    return load().moe_route(_ref(cfg), _ref(wts), _ptr(x), int(n), _ptr(idx),
                            _ptr(w), _ptr(logits), _ptr(ws), int(ws_bytes), _stream(stream))


def moe_experts(cfg, wts, x, n, idx, w, out, ws, ws_bytes, stream=None) -> int:
    return load().moe_experts(_ref(cfg), _ref(wts), _ptr(x), int(n), _ptr(idx),
                              _ptr(w), _ptr(out), _ptr(ws), int(ws_bytes), _stream(stream))


def moe_forward(cfg, wts, x, n, out, idx, w, ws, ws_bytes, stream=None) -> int:
    return load().moe_forward(_ref(cfg), _ref(wts), _ptr(x), int(n), _ptr(out),
                              _ptr(idx), _ptr(w), _ptr(ws), int(ws_bytes), _stream(stream))


def moe_forward_timed(cfg, wts, x, n, out, idx, w, ws, ws_bytes, stream, events):
    """``events``: a list of raw cudaEvent_t handles (ints).  Returns
    (status, markers reached)."""
    arr = (ctypes.c_void_p * max(1, len(events)))(*events)
    nm = ctypes.c_int32(0)
    s = load().moe_forward_timed(_ref(cfg), _ref(wts), _ptr(x), int(n), _ptr(out), _ptr(idx),
                                 _ptr(w), _ptr(ws), int(ws_bytes), _stream(stream), arr,
                                 len(events), ctypes.byref(nm))
    return s, nm.value


def moe_forward_static_ws(cfg, wts, x, n, out, idx, w, stream=None) -> int:
    """moe_forward with the library's static device workspace (no ws argument)."""
    return load().moe_forward_static_ws(_ref(cfg), _ref(wts), _ptr(x), int(n), _ptr(out), _ptr(idx),
                                        _ptr(w), _stream(stream))


def moe_static_workspace_check(stream=None):
    """(status, device error word, static workspace device address) of
    moe_forward_static_ws on the current device; reads and clears the word,
    syncing the stream."""
    v = ctypes.c_int32(0)
    addr = ctypes.c_void_p(None)
    s = load().moe_static_workspace_check(ctypes.byref(v), ctypes.byref(addr), _stream(stream))
    return s, v.value, addr.value


def moe_workspace_check(ws, ws_bytes, stream=None):
    """(status, device error word); reads and clears the word, syncing the stream."""
    v = ctypes.c_int32(0)
    s = load().moe_workspace_check(_ptr(ws), int(ws_bytes), ctypes.byref(v), _stream(stream))
    return s, v.value


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_abi_version() -> int:
    return load().moe_abi_version()


class MoeError(RuntimeError):
    pass


def check(status: int) -> None:
    if status != MOE_OK:
        raise MoeError(moe_status_string(status))
