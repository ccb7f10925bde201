"""ctypes binding of libmoe.so (include/moe.h), same names as the C ABI.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  torch supplies device memory and the current CUDA stream.  Importing
this module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m mixture_experts_layer_85_b300.build`")

_lib = ctypes.CDLL(LIB_PATH)

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, \
    MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_BOUNDS, MOE_ERR_DEVICE_RANGE = range(8)
MOE_F32, MOE_BF16, MOE_FP8_E4M3 = 0, 1, 2
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_TOPK_GREEDY, MOE_TOPK_GROUP_LIMITED = 0, 1
MOE_GROUP_MAX, MOE_GROUP_SUM_TOP = 0, 1

EXPORTED = ["moe_workspace_size", "moe_packed_size", "moe_prepack_experts", "moe_gate_topk", "moe_permute",
            "moe_grouped_swiglu", "moe_combine", "moe_forward", "moe_get_device_status", "moe_status_string",
            "moe_launch_count", "moe_forward_kernel_count", "moe_profile_arm", "moe_forward_stage_name",
            "moe_permute_noalloc", "moe_balance_update", "moe_backward_workspace_size", "moe_backward",
            "moe_debug_inject"]
MOE_FORWARD_STAGES = 4
MOE_DEBUG_WAIT_LIMIT_NS, MOE_DEBUG_STALL_GEMM2 = 0, 1


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32), ("I", ctypes.c_int32),
                ("k", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("score_fn", ctypes.c_int32),
                ("topk_method", ctypes.c_int32), ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("group_score", ctypes.c_int32), ("group_top", ctypes.c_int32), ("norm_topk", ctypes.c_int32),
                ("routed_scaling_factor", ctypes.c_float), ("act_dtype", ctypes.c_int32),
                ("gate_w_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("expert_w_dtype", ctypes.c_int32)]


_P = ctypes.c_void_p
_CFG = ctypes.POINTER(moe_config)
_SZ = ctypes.c_size_t
_sigs = {
    "moe_workspace_size": [_CFG, ctypes.POINTER(_SZ)],
    "moe_packed_size": [_CFG, ctypes.POINTER(_SZ)],
    "moe_prepack_experts": [_CFG, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_gate_topk": [_CFG, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_permute": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_grouped_swiglu": [_CFG, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_combine": [_CFG, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_forward": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "moe_get_device_status": [_P, _P, ctypes.POINTER(ctypes.c_int32)],
    "moe_status_string": [ctypes.c_int],
    "moe_launch_count": [],
    "moe_forward_kernel_count": [_CFG],
    "moe_profile_arm": [ctypes.POINTER(_P), ctypes.c_int32],
    "moe_forward_stage_name": [ctypes.c_int32],
    "moe_permute_noalloc": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_balance_update": [_CFG, _P, _P, ctypes.c_float, _P, _P, _P],
    "moe_backward_workspace_size": [_CFG, ctypes.POINTER(_SZ)],
    "moe_backward": [_CFG] + [_P] * 19 + [_SZ, _P],
    "moe_debug_inject": [ctypes.c_int32, ctypes.c_int64],
}
for _name, _args in _sigs.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_lib.moe_status_string.restype = ctypes.c_char_p
_lib.moe_launch_count.restype = ctypes.c_uint64
_lib.moe_forward_kernel_count.restype = ctypes.c_int32
_lib.moe_forward_stage_name.restype = ctypes.c_char_p


class MoeError(RuntimeError):
    def __init__(self, code: int, call: str):
        self.code = code
        super().__init__(f"{call} -> {status_string(code)}")


def status_string(code: int) -> str:
    return _lib.moe_status_string(int(code)).decode()


def _check(code: int, call: str):
    if code != MOE_OK:
        raise MoeError(code, call)


def make_config(wl, T: Optional[int] = None) -> moe_config:
    """moe_config of a workload (see inputs.Workload)."""
    c = moe_config()
    c.T = wl.T if T is None else T
    c.d, c.E, c.I, c.k, c.n_shared = wl.d, wl.E, wl.I, wl.k, wl.n_shared
    c.score_fn = MOE_SCORE_SOFTMAX if wl.score_fn == "softmax" else MOE_SCORE_SIGMOID
    c.topk_method = MOE_TOPK_GREEDY if wl.topk_method == "greedy" else MOE_TOPK_GROUP_LIMITED
    c.n_group, c.topk_group = wl.n_group, wl.topk_group
    c.group_score = MOE_GROUP_MAX if wl.group_score == "max" else MOE_GROUP_SUM_TOP
    c.group_top = wl.group_top
    c.norm_topk = 1 if wl.norm_topk else 0
    c.routed_scaling_factor = wl.routed_scaling_factor
    c.act_dtype = MOE_BF16 if wl.act_dtype == "bf16" else MOE_F32
    c.gate_w_dtype = MOE_BF16 if wl.gate_w_dtype == "bf16" else MOE_F32
    c.out_dtype = MOE_BF16 if wl.out_dtype == "bf16" else MOE_F32
    c.expert_w_dtype = MOE_FP8_E4M3 if wl.expert_w_dtype == "fp8" else c.act_dtype
    return c


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def moe_workspace_size(cfg: moe_config) -> int:
    n = _SZ(0)
    _check(_lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_packed_size(cfg: moe_config) -> int:
    n = _SZ(0)
    _check(_lib.moe_packed_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_packed_size")
    return n.value


def moe_prepack_experts(cfg, W1, W3, W2, Ws1, Ws3, Ws2, packed, stream=None):
    _check(_lib.moe_prepack_experts(ctypes.byref(cfg), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(Ws1), _ptr(Ws3),
                                    _ptr(Ws2), _ptr(packed), packed.numel() * packed.element_size(),
                                    _stream(stream)), "moe_prepack_experts")


def moe_gate_topk(cfg, x, Wg, bias, idx, w, ws, stream=None):
    _check(_lib.moe_gate_topk(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(bias), _ptr(idx), _ptr(w), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "moe_gate_topk")


def moe_permute(cfg, x, idx, counts, offsets, row2tok, tok2row, x_perm, ws, stream=None):
    _check(_lib.moe_permute(ctypes.byref(cfg), _ptr(x), _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(row2tok),
                            _ptr(tok2row), _ptr(x_perm), _ptr(ws), ws.numel() * ws.element_size(),
                            _stream(stream)), "moe_permute")


def moe_grouped_swiglu(cfg, x_perm, offsets, x, packed, y_perm, y_shared, ws, stream=None):
    _check(_lib.moe_grouped_swiglu(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(x), _ptr(packed),
                                   _ptr(y_perm), _ptr(y_shared), _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)), "moe_grouped_swiglu")


def moe_combine(cfg, y_perm, y_shared, tok2row, w, out, ws, stream=None):
    _check(_lib.moe_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(y_shared), _ptr(tok2row), _ptr(w), _ptr(out),
                            _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_combine")


def moe_forward(cfg, x, Wg, bias, packed, out, ws, idx_out=None, w_out=None, counts_out=None, stream=None):
    _check(_lib.moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(bias), _ptr(packed), _ptr(out),
                            _ptr(idx_out), _ptr(w_out), _ptr(counts_out), _ptr(ws), ws.numel() * ws.element_size(),
                            _stream(stream)), "moe_forward")


def moe_permute_noalloc(cfg, x, idx, counts, offsets, row2tok, tok2row, x_perm, device_status=None, stream=None):
    """moe_permute without a workspace: scratch in the library's fixed device array."""
    _check(_lib.moe_permute_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(idx), _ptr(counts), _ptr(offsets),
                                    _ptr(row2tok), _ptr(tok2row), _ptr(x_perm), _ptr(device_status),
                                    _stream(stream)), "moe_permute_noalloc")


def moe_balance_update(cfg, counts, bias, gamma: float, stats=None, device_status=None, stream=None):
    """Aux-loss-free bias update from per-expert counts (bias updated in place)."""
    _check(_lib.moe_balance_update(ctypes.byref(cfg), _ptr(counts), _ptr(bias), float(gamma), _ptr(stats),
                                   _ptr(device_status), _stream(stream)), "moe_balance_update")


def moe_backward_workspace_size(cfg: moe_config) -> int:
    n = _SZ(0)
    _check(_lib.moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_backward_workspace_size")
    return n.value


def moe_backward(cfg, x, Wg, bias, W1, W3, W2, Ws1, Ws3, Ws2, dout, dx, dWg, dW1, dW3, dW2, dWs1, dWs3, dWs2, ws,
                 stream=None):
    """Gradients of <dout, out> (fp32 outputs written in place); synchronises the stream once."""
    _check(_lib.moe_backward(ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(bias), _ptr(W1), _ptr(W3), _ptr(W2),
                             _ptr(Ws1), _ptr(Ws3), _ptr(Ws2), _ptr(dout), _ptr(dx), _ptr(dWg), _ptr(dW1), _ptr(dW3),
                             _ptr(dW2), _ptr(dWs1), _ptr(dWs3), _ptr(dWs2), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream)),
           "moe_backward")


def moe_get_device_status(ws, stream=None) -> tuple:
    """(status code, raw device status word); synchronises the stream."""
    word = ctypes.c_int32(0)
    code = _lib.moe_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(word))
    return code, word.value


def moe_status_string(code: int) -> str:
    return status_string(code)


def moe_launch_count() -> int:
    return int(_lib.moe_launch_count())


def moe_forward_kernel_count(cfg) -> int:
    return int(_lib.moe_forward_kernel_count(ctypes.byref(cfg)))


_armed = None


def moe_profile_arm(events) -> None:
    """Arms stage timing with a list of torch.cuda.Event (timing enabled); None
    disarms.  Each moe_forward uses MOE_FORWARD_STAGES + 1 of them."""
    global _armed
    if events is None:
        _check(_lib.moe_profile_arm(None, 0), "moe_profile_arm")
        _armed = None
        return
    for ev in events:          # torch creates the CUDA event lazily
        if ev.cuda_event == 0:
            ev.record()
    arr = (_P * len(events))(*[ev.cuda_event for ev in events])
    _armed = (arr, events)     # keep the handle array alive while armed
    _check(_lib.moe_profile_arm(arr, len(events)), "moe_profile_arm")


def moe_forward_stage_name(i: int) -> Optional[str]:
    n = _lib.moe_forward_stage_name(int(i))
    return None if n is None else n.decode()


def moe_debug_inject(what: int, value: int):
    """Test-only fault injection of the expert kernel's bounded waits."""
    _check(_lib.moe_debug_inject(int(what), int(value)), "moe_debug_inject")


def raw_call(name: str, *args) -> int:
    """The C function itself (for tests of argument validation)."""
    return getattr(_lib, name)(*args)
