"""ctypes binding of the C ABI in include/moe.h (argument marshalling only).

The functions below carry the C names and forward to libmoe_b300.so; every step
of the layer runs in that library's CUDA kernels.  There is no fallback: if the
library is missing and cannot be built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

_i32, _u32, _f32, _vp = ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_void_p

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5

MOE_ACT_RELU, MOE_ACT_GELU_TANH, MOE_ACT_GELU_ERF, MOE_ACT_SWIGLU = 0, 1, 2, 3
MOE_F32, MOE_BF16 = 0, 1
MOE_FLAG_FFMA_EXPERTS = 1
MOE_FLAG_FFMA_ROUTER = 2
MOE_FLAG_UNFUSED_EXPERTS = 4
MOE_FLAG_TRAINING = 8
MOE_WEIGHTS_DTYPE, MOE_WEIGHTS_INT8, MOE_WEIGHTS_INT4 = 0, 1, 2
MOE_INT4_GROUP = 128
MOE_MAX_EXPERTS = 512
MOE_MAX_TOPK = 32
MOE_NOALLOC_MAX_SLOTS = 131072
MOE_EP_MAX_RANKS = 16


class moe_params_t(ctypes.Structure):
    _fields_ = [("T", _i32), ("d_model", _i32), ("d_ff", _i32), ("E", _i32), ("k", _i32),
                ("n_shared", _i32), ("capacity_factor", _f32), ("renormalize", _i32),
                ("residual_mode", _i32), ("act", _i32), ("dtype", _i32), ("flags", _u32),
                ("noisy_gating", _i32), ("noise_min_std", _f32), ("weight_format", _i32)]


class moe_inputs_t(ctypes.Structure):
    _fields_ = [("x", _vp), ("W_gate", _vp), ("b_gate", _vp), ("W1", _vp), ("W3", _vp),
                ("W2", _vp), ("b1", _vp), ("b2", _vp), ("W_noise", _vp), ("b_noise", _vp),
                ("noise_eps", _vp), ("W1_scale", _vp), ("W3_scale", _vp), ("W2_scale", _vp),
                ("router_weights", _vp)]


class moe_outputs_t(ctypes.Structure):
    _fields_ = [("y", _vp), ("expert_idx", _vp), ("gates", _vp), ("counts", _vp),
                ("dropped", _vp), ("aux", _vp), ("logits", _vp), ("probs", _vp),
                ("perm_row", _vp)]


class moe_grads_t(ctypes.Structure):
    _fields_ = [("dx", _vp), ("dW_gate", _vp), ("db_gate", _vp), ("dW1", _vp), ("dW3", _vp),
                ("dW2", _vp), ("db1", _vp), ("db2", _vp), ("dW_noise", _vp), ("db_noise", _vp)]


_P = ctypes.POINTER
_STAGE_ARGS = [_P(moe_params_t), _P(moe_inputs_t), _P(moe_outputs_t), _vp, ctypes.c_size_t, _vp]
STAGES = ("moe_forward", "moe_router", "moe_dispatch", "moe_grouped_gemm", "moe_combine")

_handle = None


def library_path() -> str:
    return _build.LIB


def load(build_if_stale: bool = True):
    """Load libmoe_b300.so (building it first if sources are newer)."""
    global _handle
    if _handle is not None:
        return _handle
    if build_if_stale and _build.needs_build():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"CUDA library missing: {_build.LIB} (run sparse_mixture_experts_scan_b300.build)")
    L = ctypes.CDLL(_build.LIB)
    L.moe_workspace_size.restype = _i32
    L.moe_workspace_size.argtypes = [_P(moe_params_t), _P(ctypes.c_size_t)]
    for name in STAGES:
        f = getattr(L, name)
        f.restype = _i32
        f.argtypes = _STAGE_ARGS
    L.moe_backward.restype = _i32
    L.moe_backward.argtypes = [_P(moe_params_t), _P(moe_inputs_t), _P(moe_outputs_t), _vp, _f32,
                               _P(moe_grads_t), _vp, ctypes.c_size_t, _vp]
    L.moe_last_device_status.restype = _i32
    L.moe_last_device_status.argtypes = [_vp, ctypes.c_size_t, _vp]
    L.moe_dispatch_positions_noalloc.restype = _i32
    L.moe_dispatch_positions_noalloc.argtypes = [_P(moe_params_t), _vp, _vp, _vp, _vp, _vp]
    L.moe_quantize_int8.restype = _i32
    L.moe_quantize_int8.argtypes = [_vp, _i32, ctypes.c_int64, _i32, _vp, _vp, _vp]
    L.moe_quantize_int4.restype = _i32
    L.moe_quantize_int4.argtypes = [_vp, _i32, ctypes.c_int64, _i32, _vp, _vp, _vp]
    L.moe_check_bounded_wait.restype = _i32
    L.moe_check_bounded_wait.argtypes = [_vp, ctypes.c_size_t, _u32, _vp]
    L.moe_kernel_launches.restype = ctypes.c_uint64
    L.moe_kernel_launches.argtypes = []
    L.moe_router_weights_size.restype = _i32
    L.moe_router_weights_size.argtypes = [_P(moe_params_t), _P(ctypes.c_size_t)]
    L.moe_prepare_router_weights.restype = _i32
    L.moe_prepare_router_weights.argtypes = [_P(moe_params_t), _vp, _vp, _vp, ctypes.c_size_t, _vp]
    L.moe_ep_workspace_size.restype = _i32
    L.moe_ep_workspace_size.argtypes = [_P(moe_params_t), _i32, _P(ctypes.c_size_t)]
    L.moe_forward_ep.restype = _i32
    L.moe_forward_ep.argtypes = [_P(moe_params_t), _i32, _P(moe_inputs_t), _P(moe_outputs_t), _vp,
                                 ctypes.c_size_t, _vp]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_status_string.argtypes = [_i32]
    _handle = L
    return L


def header_functions() -> list[str]:
    """Names of the functions include/moe.h declares."""
    path = os.path.join(_build.INCLUDE, "moe.h")
    with open(path) as f:
        text = f.read()
    return re.findall(r"^\s*(?:const\s+char\s*\*|moe_status_t|uint64_t)\s+(moe_\w+)\s*\(", text, re.M)


# ---- the C entry points, same names ---------------------------------------

def moe_workspace_size(params: moe_params_t):
    n = ctypes.c_size_t(0)
    st = load().moe_workspace_size(ctypes.byref(params), ctypes.byref(n))
    return st, n.value


def _stage(name, params, inputs, outputs, workspace, workspace_bytes, stream):
    f = getattr(load(), name)
    return f(ctypes.byref(params), ctypes.byref(inputs), ctypes.byref(outputs),
             _vp(workspace), ctypes.c_size_t(workspace_bytes), _vp(stream))


def moe_forward(params, inputs, outputs, workspace, workspace_bytes, stream):
    return _stage("moe_forward", params, inputs, outputs, workspace, workspace_bytes, stream)


def moe_router(params, inputs, outputs, workspace, workspace_bytes, stream):
    return _stage("moe_router", params, inputs, outputs, workspace, workspace_bytes, stream)


def moe_dispatch(params, inputs, outputs, workspace, workspace_bytes, stream):
    return _stage("moe_dispatch", params, inputs, outputs, workspace, workspace_bytes, stream)


def moe_grouped_gemm(params, inputs, outputs, workspace, workspace_bytes, stream):
    return _stage("moe_grouped_gemm", params, inputs, outputs, workspace, workspace_bytes, stream)


def moe_combine(params, inputs, outputs, workspace, workspace_bytes, stream):
    return _stage("moe_combine", params, inputs, outputs, workspace, workspace_bytes, stream)


def moe_backward(params, inputs, outputs, dy, d_aux, grads, workspace, workspace_bytes, stream):
    return load().moe_backward(ctypes.byref(params), ctypes.byref(inputs), ctypes.byref(outputs), _vp(dy),
                               _f32(d_aux), ctypes.byref(grads), _vp(workspace),
                               ctypes.c_size_t(workspace_bytes), _vp(stream))


def moe_router_weights_size(params: moe_params_t):
    n = ctypes.c_size_t(0)
    st = load().moe_router_weights_size(ctypes.byref(params), ctypes.byref(n))
    return st, n.value


def moe_prepare_router_weights(params, W_gate, W_noise, prepared, prepared_bytes, stream):
    return load().moe_prepare_router_weights(ctypes.byref(params), _vp(W_gate), _vp(W_noise), _vp(prepared),
                                             ctypes.c_size_t(prepared_bytes), _vp(stream))


def moe_ep_workspace_size(params: moe_params_t, G: int):
    n = ctypes.c_size_t(0)
    st = load().moe_ep_workspace_size(ctypes.byref(params), _i32(G), ctypes.byref(n))
    return st, n.value


def moe_forward_ep(params, G, inputs, outputs, workspace, workspace_bytes, stream):
    return load().moe_forward_ep(ctypes.byref(params), _i32(G), ctypes.byref(inputs), ctypes.byref(outputs),
                                 _vp(workspace), ctypes.c_size_t(workspace_bytes), _vp(stream))


def moe_dispatch_positions_noalloc(params, expert_idx, counts, dropped, perm_row, stream):
    return load().moe_dispatch_positions_noalloc(ctypes.byref(params), _vp(expert_idx), _vp(counts),
                                                 _vp(dropped), _vp(perm_row), _vp(stream))


def moe_last_device_status(workspace, workspace_bytes, stream):
    return load().moe_last_device_status(_vp(workspace), ctypes.c_size_t(workspace_bytes), _vp(stream))


def moe_quantize_int8(w, dtype, rows, cols, q, scale, stream):
    return load().moe_quantize_int8(_vp(w), _i32(dtype), ctypes.c_int64(rows), _i32(cols), _vp(q), _vp(scale),
                                    _vp(stream))


def moe_quantize_int4(w, dtype, rows, cols, q, scale, stream):
    return load().moe_quantize_int4(_vp(w), _i32(dtype), ctypes.c_int64(rows), _i32(cols), _vp(q), _vp(scale),
                                    _vp(stream))


def moe_check_bounded_wait(workspace, workspace_bytes, timeout_us, stream):
    return load().moe_check_bounded_wait(_vp(workspace), ctypes.c_size_t(workspace_bytes), _u32(timeout_us),
                                         _vp(stream))


def moe_kernel_launches() -> int:
    return int(load().moe_kernel_launches())


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()
