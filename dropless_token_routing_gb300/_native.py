"""ctypes binding of ``libmoe.so`` (the C ABI declared in include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Importing this module fails loudly if the library is not built.
"""
from __future__ import annotations

import ctypes
import os
import re

from .builder import INCLUDE, LIB

if not os.path.exists(LIB):
    raise ImportError(
        f"{LIB} is missing: build the CUDA library first "
        "(python -m dropless_token_routing_gb300.builder)")

_lib = ctypes.CDLL(LIB)

c_int, c_int32, c_int64, c_size_t, c_void_p, c_uint64 = (
    ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_uint64)

MOE_F32, MOE_BF16 = 0, 1

STATUS = {
    0: "MOE_OK", -1: "MOE_ERR_NULL_POINTER", -2: "MOE_ERR_MISALIGNED", -3: "MOE_ERR_BAD_DIMS",
    -4: "MOE_ERR_BAD_TOPK", -5: "MOE_ERR_UNSUPPORTED_DTYPE", -6: "MOE_ERR_WORKSPACE_TOO_SMALL",
    -7: "MOE_ERR_LAUNCH", -8: "MOE_ERR_CUDA", -9: "MOE_ERR_UNSUPPORTED_DEVICE",
    -100: "MOE_ERR_DEVICE_EXPERT_ID", -101: "MOE_ERR_DEVICE_TIMEOUT",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}


class MoeError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call} -> {STATUS.get(status, status)}: {status_string(status)}")


class MoeDims(ctypes.Structure):
    _fields_ = [("T", c_int64), ("d", c_int32), ("E", c_int32), ("k", c_int32), ("f", c_int32),
                ("S", c_int32), ("f_s", c_int32), ("dtype", c_int32), ("capacity", c_int32),
                ("rearrange", c_int32)]


class LayerParams(ctypes.Structure):
    _fields_ = [("w_r", c_void_p), ("bias", c_void_p), ("w13", c_void_p), ("w2", c_void_p),
                ("ws13", c_void_p), ("ws2", c_void_p)]


class LayerSaved(ctypes.Structure):
    _fields_ = [("logits", c_void_p), ("topk_idx", c_void_p), ("topk_w", c_void_p),
                ("counts", c_void_p), ("offsets", c_void_p), ("dest", c_void_p),
                ("row_src", c_void_p), ("w_perm", c_void_p), ("x_perm", c_void_p), ("z", c_void_p),
                ("h", c_void_p), ("z_sh", c_void_p), ("h_sh", c_void_p)]


class TraceEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", c_int64), ("total_ms", ctypes.c_double)]


class LayerGrads(ctypes.Structure):
    _fields_ = [("dx", c_void_p), ("dw13", c_void_p), ("dw2", c_void_p), ("dws13", c_void_p),
                ("dws2", c_void_p), ("dw_r", c_void_p), ("dlogits", c_void_p)]


P = c_void_p
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [c_int]),
    "moe_workspace_bytes": (c_size_t, [ctypes.POINTER(MoeDims)]),
    "moe_workspace_init": (c_int, [P, c_size_t, ctypes.POINTER(MoeDims), P]),
    "moe_get_device_error": (c_int, [P, P, ctypes.POINTER(c_int)]),
    "moe_router_logits": (c_int, [P, P, ctypes.POINTER(MoeDims), P, P, c_size_t, P]),
    "moe_route_topk": (c_int, [P, P, c_int64, c_int32, c_int32, P, P, P, P, c_size_t, P]),
    "moe_permute": (c_int, [P, P, P, ctypes.POINTER(MoeDims), P, P, P, P, P, P, c_size_t, P]),
    "moe_permute_rows": (c_int, [P, P, ctypes.POINTER(MoeDims), P, P]),
    "moe_permute_noalloc": (c_int, [P, P, P, ctypes.POINTER(MoeDims), P, P, P, P, P, P, P]),
    "moe_grouped_swiglu_fwd": (c_int, [P, P, P, P, P, P, P, ctypes.POINTER(MoeDims), P, P, P, P, P,
                                       P, P, c_size_t, P]),
    "moe_unpermute_combine": (c_int, [P, P, P, P, ctypes.POINTER(MoeDims), P, P]),
    "moe_grouped_bwd_dx": (c_int, [P, P, P, P, P, P, P, P, P, P, P, ctypes.POINTER(MoeDims), P, P,
                                   P, P, P, P, P, P, c_size_t, P]),
    "moe_grouped_bwd_dw": (c_int, [P, P, P, P, P, P, P, P, P, ctypes.POINTER(MoeDims), P, P, P, P,
                                   P, c_size_t, P]),
    "moe_route_topk_bwd": (c_int, [P, P, P, c_int64, c_int32, c_int32, P, P]),
    "moe_route_balance": (c_int, [P, P, P, c_int64, c_int32, c_int32, ctypes.c_float, P, P, P, c_size_t, P]),
    "moe_route_topk_balance": (c_int, [P, P, c_int64, c_int32, c_int32, ctypes.c_float, P, P, P, P, P, P,
                                       c_size_t, P]),
    "moe_route_balance_bwd": (c_int, [P, P, P, c_int64, c_int32, c_int32, ctypes.c_float, ctypes.c_float, P, P]),
    "moe_route_balance_seq": (c_int, [P, P, P, c_int64, c_int32, c_int32, c_int64, ctypes.c_float, P, P, P, P,
                                      c_size_t, P]),
    "moe_route_balance_seq_bwd": (c_int, [P, P, P, c_int64, c_int32, c_int32, c_int64, c_int64,
                                          ctypes.c_float, ctypes.c_float, P, P]),
    "moe_layer_fwd": (c_int, [ctypes.POINTER(LayerParams), P, P, ctypes.POINTER(MoeDims),
                              ctypes.POINTER(LayerSaved), P, P, c_size_t, P]),
    "moe_layer_bwd": (c_int, [ctypes.POINTER(LayerParams), ctypes.POINTER(LayerSaved), P, P,
                              ctypes.POINTER(MoeDims), ctypes.POINTER(LayerGrads), P, c_size_t, P]),
    "moe_debug_timeout_probe": (c_int, [P, c_size_t, c_uint64, P]),
    "moe_trace_enable": (c_int, [c_int]),
    "moe_trace_read": (c_int, [ctypes.POINTER(TraceEntry), c_int, ctypes.POINTER(c_int)]),
}

for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def header_functions():
    """Names of the functions include/moe.h declares."""
    text = open(os.path.join(INCLUDE, "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def lib():
    return _lib


def status_string(s: int) -> str:
    return _lib.moe_status_string(int(s)).decode()


def trace_enable(on: bool) -> None:
    check(_lib.moe_trace_enable(1 if on else 0), "moe_trace_enable")


def trace_read() -> dict:
    """{phase: (launches, total_ms)} of the launches recorded since trace_enable(True)."""
    buf = (TraceEntry * 64)()
    n = c_int(0)
    check(_lib.moe_trace_read(buf, 64, ctypes.byref(n)), "moe_trace_read")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n.value)}


def check(status: int, call: str):
    if status != 0:
        raise MoeError(status, call)
