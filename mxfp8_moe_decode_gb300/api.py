"""Python binding of the C ABI, on torch tensors (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
checks tensor shapes / dtypes / devices (the kernels' loads are unbounded, so
a mismatch must be caught here, as the runner page's ``_check_tensors``
does) and passes raw pointers and the current stream.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import MoeConfig, MoeDebug, MoeWeights, check

WEIGHT_KEYS = ("norm_w", "gate_w", "bias", "w13", "w13_s", "w2", "w2_s",
               "sw13", "sw13_s", "sw2", "sw2_s")


def _u8(t: torch.Tensor) -> torch.Tensor:
    fp4x2 = getattr(torch, "float4_e2m1fn_x2", None)
    return t.view(torch.uint8) if t.dtype in (torch.float8_e4m3fn, fp4x2) else t


def expected_shapes(hidden: int, experts: int, inter: int, shared_inter: int,
                    routed: str = "e4m3") -> dict:
    """Weight shapes and dtypes; ``routed="e2m1"``: MXFP4 routed experts (E2M1
    pairs, one code per row per 32 columns)."""
    h, e, i, s = hidden, experts, inter, shared_inter
    if routed == "e2m1":
        fp4 = {"w13": ((e, 2 * i, h // 2), torch.uint8),
               "w13_s": ((e, 2 * i, h // 32), torch.uint8),
               "w2": ((e, h, i // 2), torch.uint8),
               "w2_s": ((e, h, i // 32), torch.uint8)}
        return {**expected_shapes(hidden, experts, inter, shared_inter), **fp4}
    if routed != "e4m3":
        raise ValueError(f"routed weights: 'e4m3' or 'e2m1', not {routed!r}")
    return {
        "norm_w": ((h,), torch.bfloat16),
        "gate_w": ((e, h), torch.bfloat16),
        "bias": ((e,), torch.float32),
        "w13": ((e, 2 * i, h), torch.uint8),
        "w13_s": ((e, 2 * i // 32, h // 32), torch.uint8),
        "w2": ((e, h, i), torch.uint8),
        "w2_s": ((e, h // 32, i // 32), torch.uint8),
        "sw13": ((2 * s, h), torch.uint8),
        "sw13_s": ((2 * s // 32, h // 32), torch.uint8),
        "sw2": ((h, s), torch.uint8),
        "sw2_s": ((h // 32, s // 32), torch.uint8),
    }


class _DeviceBytes:
    """Raw device memory exposed through __cuda_array_interface__ (read by torch)."""

    def __init__(self, ptr: int, nbytes: int):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (ptr, False), "version": 3}


def attn_seam_x8(x: torch.Tensor, norm_w: torch.Tensor, eps: float = 1e-6,
                 x8: torch.Tensor | None = None, codes: torch.Tensor | None = None,
                 ys: torch.Tensor | None = None):
    """Attention-seam MXFP8 of bf16 rows x [M, H] (``moe_attn_seam_x8``): the
    fp32 RMSNorm with ``norm_w`` bf16 [H], quantised from its fp32 values.

    Returns (x8 uint8 [M, H], codes uint8 [M, H/32], ys) where ys is the fp32
    norm output [M, H] if a tensor was passed for it, else None. Outputs not
    passed are allocated here (on x's device); the kernel runs on the current
    stream.
    """
    if x.dim() != 2 or x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA bf16 [M, H] tensor")
    M, H = x.shape
    if (norm_w.shape != (H,) or norm_w.dtype != torch.bfloat16 or norm_w.device != x.device
            or not norm_w.is_contiguous()):
        raise ValueError("norm_w must be a contiguous bf16 [H] tensor on x's device")
    if H % 32:
        raise ValueError("H must be a multiple of 32")
    want = {"x8": ((M, H), torch.uint8), "codes": ((M, H // 32), torch.uint8),
            "ys": ((M, H), torch.float32)}
    got = {"x8": x8, "codes": codes, "ys": ys}
    for k, t in got.items():
        if t is not None and (tuple(t.shape) != want[k][0] or t.dtype != want[k][1]
                              or t.device != x.device or not t.is_contiguous()):
            raise ValueError(f"{k} must be a contiguous {want[k][1]} {want[k][0]} tensor on x's device")
    if x8 is None:
        x8 = torch.empty((M, H), dtype=torch.uint8, device=x.device)
    if codes is None:
        codes = torch.empty((M, H // 32), dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        stream = torch.cuda.current_stream().cuda_stream
    check(_lib.lib().moe_attn_seam_x8(
        x.data_ptr(), norm_w.data_ptr(), M, H, float(eps), x8.data_ptr(), codes.data_ptr(),
        ys.data_ptr() if ys is not None else None, stream), "moe_attn_seam_x8")
    return x8, codes, ys


def kernel_names() -> list[str]:
    L = _lib.lib()
    return [L.moe_kernel_name(i).decode() for i in range(L.moe_kernel_count())]


class MoeDecode:
    """One MoE layer's decode step on one GPU.

    weights: dict with the tensors of ``WEIGHT_KEYS`` on the target device
    (E4M3 tensors as uint8 or float8_e4m3fn; with ``routed="e2m1"`` the routed
    w13 / w2 as uint8 E2M1 pairs or float4_e2m1fn_x2, their scales per row).
    The handle keeps references to them; they must not change while it lives
    (the E8M0 scales are packed at creation).
    """

    def __init__(self, hidden: int, experts: int, topk: int, inter: int, weights: dict,
                 shared_inter: int | None = None, max_tokens: int = 48, eps: float = 1e-6,
                 device=None, routed: str = "e4m3"):
        L = _lib.lib()
        shared_inter = inter if shared_inter is None else shared_inter
        dev = torch.device(device) if device is not None else weights["gate_w"].device
        if dev.type != "cuda":
            raise ValueError("MoeDecode needs CUDA tensors")
        want = expected_shapes(hidden, experts, inter, shared_inter, routed)
        self._w = {}
        for k, (shape, dtype) in want.items():
            t = weights[k]
            t = _u8(t)
            if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous() \
                    or t.device != dev:
                raise ValueError(f"weight {k}: {tuple(t.shape)} {t.dtype} {t.device}, "
                                 f"want {shape} {dtype} contiguous on {dev}")
            self._w[k] = t
        self.hidden, self.experts, self.topk, self.inter = hidden, experts, topk, inter
        self.max_tokens = max_tokens
        self.device = dev
        fmt = _lib.MOE_ROUTED_E2M1 if routed == "e2m1" else _lib.MOE_ROUTED_E4M3
        cfg = MoeConfig(hidden, experts, topk, inter, shared_inter, max_tokens, eps, fmt)
        wt = MoeWeights(*[self._w[k].data_ptr() for k in WEIGHT_KEYS])
        h = ctypes.c_void_p()
        with torch.cuda.device(dev):
            check(L.moe_create(ctypes.byref(cfg), ctypes.byref(wt), dev.index or 0,
                               ctypes.byref(h)), "moe_create")
        self._h = h
        self._events = None

    # ------------------------------------------------------------ steps
    def step(self, x: torch.Tensor, out: torch.Tensor | None = None, debug: dict | None = None,
             stream: torch.cuda.Stream | None = None) -> torch.Tensor:
        """x bf16 [M, H] on the device -> out bf16 [M, H] (enqueued on the stream)."""
        if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != self.hidden \
                or not x.is_contiguous() or x.device != self.device:
            raise ValueError(f"x: {tuple(x.shape)} {x.dtype} {x.device}")
        m = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        elif out.shape != x.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() \
                or out.device != self.device:
            raise ValueError(f"out: {tuple(out.shape)} {out.dtype}")
        dbg = None
        if debug:
            dbg = MoeDebug(*[self._dbg_ptr(debug, k, m) for k in
                             ("normed", "x8", "x8_codes", "topk_ids", "topk_w", "logits")])
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        code = _lib.lib().moe_decode_step(self._h, x.data_ptr(), m, out.data_ptr(),
                                          ctypes.c_void_p(st.cuda_stream),
                                          ctypes.byref(dbg) if dbg is not None else None)
        check(code, "moe_decode_step")
        return out

    def _dbg_ptr(self, debug: dict, key: str, m: int):
        t = debug.get(key)
        if t is None:
            return None
        shapes = {"normed": ((m, self.hidden), torch.bfloat16),
                  "x8": ((m, self.hidden), torch.uint8),
                  "x8_codes": ((m, self.hidden // 32), torch.uint8),
                  "topk_ids": ((m, self.topk), torch.int32),
                  "topk_w": ((m, self.topk), torch.float32),
                  "logits": ((m, self.experts), torch.float32)}
        shape, dtype = shapes[key]
        if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous() \
                or t.device != self.device:
            raise ValueError(f"debug {key}: {tuple(t.shape)} {t.dtype}, want {shape} {dtype}")
        return t.data_ptr()

    def debug_buffers(self, m: int) -> dict:
        d = self.device
        return {"normed": torch.empty(m, self.hidden, dtype=torch.bfloat16, device=d),
                "x8": torch.empty(m, self.hidden, dtype=torch.uint8, device=d),
                "x8_codes": torch.empty(m, self.hidden // 32, dtype=torch.uint8, device=d),
                "topk_ids": torch.empty(m, self.topk, dtype=torch.int32, device=d),
                "topk_w": torch.empty(m, self.topk, dtype=torch.float32, device=d),
                "logits": torch.empty(m, self.experts, dtype=torch.float32, device=d)}

    # ------------------------------------------------------------ status
    def status(self) -> int:
        return _lib.lib().moe_status(self._h)

    def clear_status(self) -> int:
        return _lib.lib().moe_clear_status(self._h)

    def test_withhold_ready(self, unit: int) -> None:
        """Test hook (``moe_test_withhold_ready``): the expert kernel's unit
        ``unit`` never reports its w13 tiles done, so the step's bounded waits
        expire (status MOE_ERR_TIMEOUT); -1 turns it off."""
        check(_lib.lib().moe_test_withhold_ready(self._h, unit), "test_withhold_ready")

    def step_launches(self, m: int) -> int:
        """Kernels one step of m tokens launches."""
        return _lib.lib().moe_step_launches(self._h, m)

    def unique_experts(self) -> int:
        v = ctypes.c_int()
        check(_lib.lib().moe_last_unique_experts(self._h, ctypes.byref(v)), "unique_experts")
        return v.value

    def scratch_region(self, region: int, dtype=torch.uint8, shape=None) -> torch.Tensor:
        """Copy of one scratch region (see MOE_REGION_* in the header), synchronous."""
        L = _lib.lib()
        ptr, nbytes = ctypes.c_void_p(), ctypes.c_size_t()
        check(L.moe_scratch_region(self._h, region, ctypes.byref(ptr), ctypes.byref(nbytes)),
              "scratch_region")
        torch.cuda.synchronize(self.device)
        dev = torch.as_tensor(_DeviceBytes(ptr.value, nbytes.value), device=self.device)
        t = dev.clone().cpu().view(dtype)
        return t if shape is None else t[: int(torch.tensor(shape).prod())].view(*shape)

    def scratch_bytes(self) -> int:
        return _lib.lib().moe_scratch_bytes(self._h)

    def set_timing_events(self, events) -> None:
        """events: moe_kernel_count()+1 torch.cuda.Event (one before each kernel and
        one after the last), or 2 (the step's start and end), or None to stop."""
        L = _lib.lib()
        if events is None:
            check(L.moe_set_timing_events(self._h, None, 0), "set_timing_events")
            self._events = None
            return
        for e in events:  # torch creates the CUDA event at its first record
            if not e.cuda_event:
                e.record(torch.cuda.current_stream(self.device))
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        check(L.moe_set_timing_events(self._h, arr, len(events)), "set_timing_events")
        self._events = (events, arr)

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.lib().moe_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
