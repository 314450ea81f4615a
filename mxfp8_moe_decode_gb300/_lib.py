"""ctypes declarations of libmoe_decode.so (include/moe_decode.h).

Only loads the in-tree library; it never builds or falls back to anything
else. If the library is missing, :func:`lib` raises.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_decode.so")

MOE_OK = 0
MOE_ERR_ARG = -1
MOE_ERR_RANGE = -2
MOE_ERR_ALIGN = -3
MOE_ERR_CUDA = -4
MOE_ERR_CAPTURE = -5
MOE_ERR_TIMEOUT = -6
MOE_ERR_UNSUPPORTED = -7
MOE_ERR_DEVICE = -8

REGION_GATHERED, REGION_H8, REGION_PARTIAL, REGION_ACTIVE, REGION_TOKPOS = range(5)


class MoeConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("experts", ctypes.c_int), ("topk", ctypes.c_int),
                ("inter", ctypes.c_int), ("shared_inter", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("eps", ctypes.c_float),
                ("routed_format", ctypes.c_int)]


MOE_ROUTED_E4M3 = 0
MOE_ROUTED_E2M1 = 1


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("norm_w", "gate_w", "bias", "w13", "w13_s", "w2", "w2_s",
                 "sw13", "sw13_s", "sw2", "sw2_s")]


class MoeDebug(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("normed", "x8", "x8_codes", "topk_ids", "topk_w", "logits")]


_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises FileNotFoundError if it was never built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise FileNotFoundError(
            f"{LIB_PATH} is missing: build it with `python -m mxfp8_moe_decode_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    L.moe_create.argtypes = [ctypes.POINTER(MoeConfig), ctypes.POINTER(MoeWeights), ip,
                             ctypes.POINTER(vp)]
    L.moe_create.restype = ip
    L.moe_decode_step.argtypes = [vp, vp, ip, vp, vp, ctypes.POINTER(MoeDebug)]
    L.moe_decode_step.restype = ip
    L.moe_status.argtypes = [vp]
    L.moe_status.restype = ip
    L.moe_clear_status.argtypes = [vp]
    L.moe_clear_status.restype = ip
    L.moe_last_unique_experts.argtypes = [vp, ctypes.POINTER(ip)]
    L.moe_last_unique_experts.restype = ip
    L.moe_set_timing_events.argtypes = [vp, ctypes.POINTER(vp), ip]
    L.moe_set_timing_events.restype = ip
    L.moe_kernel_count.argtypes = []
    L.moe_kernel_count.restype = ip
    L.moe_kernel_name.argtypes = [ip]
    L.moe_kernel_name.restype = ctypes.c_char_p
    L.moe_step_launches.argtypes = [vp, ip]
    L.moe_step_launches.restype = ip
    L.moe_scratch_region.argtypes = [vp, ip, ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_size_t)]
    L.moe_scratch_region.restype = ip
    L.moe_scratch_bytes.argtypes = [vp]
    L.moe_scratch_bytes.restype = ctypes.c_size_t
    L.moe_strerror.argtypes = [ip]
    L.moe_strerror.restype = ctypes.c_char_p
    L.moe_destroy.argtypes = [vp]
    L.moe_destroy.restype = None
    L.moe_attn_seam_x8.argtypes = [vp, vp, ip, ip, ctypes.c_float, vp, vp, vp, vp]
    L.moe_attn_seam_x8.restype = ip
    L.moe_test_withhold_ready.argtypes = [vp, ip]
    L.moe_test_withhold_ready.restype = ip
    L.moe_route_static.argtypes = [vp, vp, vp, ip, ip, ip, ip, vp, vp, vp]
    L.moe_route_static.restype = ip
    L.moe_route_static_status.argtypes = [vp]
    L.moe_route_static_status.restype = ip
    _LIB = L
    return L


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = lib().moe_strerror(code).decode() if _LIB is not None else str(code)
        super().__init__(f"{what}: {msg} ({code})")


def check(code: int, what: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, what)
