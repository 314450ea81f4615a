"""Seeded synthetic inputs for the MoE decode step.

This module only draws inputs: it holds none of the step's arithmetic (no
norm, no MXFP8 activation quantisation, no routing, no expert math). Both the
CUDA path's tests and the CPU oracle take their inputs from here.

Draw recipe (per workload; all tensors are inputs, identical for every
consumer):

* small tensors on the host with numpy's PCG64, one stream per tensor and
  per token row, so a row can be redrawn alone:
  - x: bf16(N(0, 1)) [M, H], row t attempt a from stream (seed, 1, t, a);
  - norm weight: bf16(1 + N(0, 0.1)) [H] (the attention seam's norm
    weight the same, from its own stream);
  - gate weight: bf16(N(0, 0.02)) [E, H];
  - bias f32 [E]: N(0, 0.01), U(-0.01, 0.01), or Zipf(s = 1.2) on a seeded
    permutation of the experts, bias[perm[r]] = C * (r + 1)^-1.2;
* expert weights with torch's generator on the target device (fast on a GPU
  for the 8 GB full-size layer), one stream per (tensor, expert):
  w ~ N(0, 0.02) fp32, then per 32 x 32 block a power-of-two scale
  2^(e - 8) where 2^(e-1) <= amax < 2^e (so every scaled value is below 256,
  inside E4M3's range), code = 127 + e - 8, bytes = torch's float8_e4m3fn
  cast of w / scale. This is a synthesis rule for the weights, which the
  pages receive already quantised; it is not the activation code of the step.
  MXFP4 routed experts (``routed="e2m1"``): per row and 32 columns a scale
  2^(e - 2), values rounded to the nearest E2M1 value (``_row_quant_fp4``).

bf16 rounding of the host draws uses torch's bfloat16 cast (round to nearest
even).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

# Zipf(s=1.2) bias scale for the 48-row full-size layer, chosen so that 48
# rows touch about 32 distinct experts (tests/golden/calibrate_zipf.py).
ZIPF_C = 5.388


@dataclass(frozen=True)
class MoeDims:
    hidden: int
    experts: int
    topk: int
    inter: int
    shared_inter: int
    max_tokens: int = 48
    eps: float = 1e-6
    routed: str = "e4m3"  # routed weights: "e4m3" (32 x 32 scales) or "e2m1" (1 x 32 per row)

    def expert_bytes(self) -> int:
        """Weight + scale bytes of one routed expert (w13 and w2)."""
        h, i = self.hidden, self.inter
        if self.routed == "e2m1":
            return (2 * i * h + h * i) // 2 + (2 * i * h + h * i) // 32
        return 2 * i * h + (2 * i // 32) * (h // 32) + h * i + (h // 32) * (i // 32)

    def shared_bytes(self) -> int:
        h, i = self.hidden, self.shared_inter
        return 2 * i * h + (2 * i // 32) * (h // 32) + h * i + (h // 32) * (i // 32)

    def router_bytes(self) -> int:
        return self.experts * self.hidden * 2 + self.experts * 4


@dataclass(frozen=True)
class Workload:
    name: str
    dims: MoeDims
    tokens: int
    seed: int
    bias: str  # "normal" | "uniform" | "zipf"
    note: str = ""
    extra: dict = field(default_factory=dict)


FULL = MoeDims(hidden=5120, experts=256, topk=8, inter=2048, shared_inter=2048)
# The runner page's layer has 384 routed experts over the same hidden size
# (gate_w [384, 5120]); its top-k and unsharded intermediate are not printed:
# these take k = 8 and I = 2048 as above, with E4M3 routed weights.
E384 = MoeDims(hidden=5120, experts=384, topk=8, inter=2048, shared_inter=2048)
# ... and its routed experts in the page's format: E2M1 pairs with one E8M0
# code per row per 32 columns (the shared expert stays E4M3, 32 x 32 blocks)
E384_FP4 = MoeDims(hidden=5120, experts=384, topk=8, inter=2048, shared_inter=2048,
                   routed="e2m1")

WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_m1", MoeDims(1024, 64, 4, 512, 512), 1, 0, "normal",
                 "tiny MoE decode step, M=1, H1024 E64 k4 I512"),
        Workload("small_m4", MoeDims(5120, 64, 4, 1024, 1024), 4, 1, "normal",
                 "small-expert layer, M=4, H5120 E64 k4 I1024"),
        Workload("full_m1", FULL, 1, 2, "uniform",
                 "full-size single-token decode, M=1, H5120 E256 k8 I2048"),
        Workload("full_m16", FULL, 16, 3, "normal",
                 "full-size batched decode, M=16"),
        Workload("full_m48_uniform", FULL, 48, 4, "uniform",
                 "max step width M=48, uniform bias"),
        Workload("full_m48_zipf", FULL, 48, 4, "zipf",
                 "max step width M=48, Zipf(1.2) bias on ~32 hot experts"),
        Workload("full_e384_m1", E384, 1, 5, "uniform",
                 "384-expert layer, single-token decode, M=1, H5120 E384 k8 I2048"),
        Workload("full_e384_m48", E384, 48, 6, "uniform",
                 "384-expert layer, M=48, uniform bias"),
        Workload("tiny_fp4", MoeDims(1024, 64, 4, 512, 512, routed="e2m1"), 1, 7, "normal",
                 "tiny layer with MXFP4 routed experts, H1024 E64 k4 I512"),
        Workload("small_fp4_m16", MoeDims(5120, 64, 4, 1024, 1024, routed="e2m1"), 16, 8,
                 "normal", "small-expert layer with MXFP4 routed experts, M=16"),
        Workload("full_e384_fp4_m1", E384_FP4, 1, 5, "uniform",
                 "384-expert layer, MXFP4 routed experts, M=1"),
        Workload("full_e384_fp4_m48", E384_FP4, 48, 6, "uniform",
                 "384-expert layer, MXFP4 routed experts, M=48, uniform bias"),
    ]
}

_TAG_X, _TAG_NORM, _TAG_GATE, _TAG_BIAS, _TAG_PERM, _TAG_ATTN_NORM = 1, 2, 3, 4, 5, 6
_T_W13, _T_W2, _T_SW13, _T_SW2 = 11, 12, 13, 14


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(key))


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def token_row(wl: Workload, t: int, attempt: int = 0) -> torch.Tensor:
    """Row t of x (bf16 [1, H], host), draw number ``attempt`` of that row."""
    r = _rng(wl.seed, _TAG_X, t, attempt).standard_normal(wl.dims.hidden, dtype=np.float32)
    return _bf16(r[None, :])


def token_rows(wl: Workload, attempts=None, m: int | None = None) -> torch.Tensor:
    """x bf16 [m, H] on the host; row t drawn from stream (seed, t, attempts[t])."""
    m = wl.tokens if m is None else m
    attempts = [0] * m if attempts is None else list(attempts)
    if m == 0:
        return torch.zeros(0, wl.dims.hidden, dtype=torch.bfloat16)
    return torch.cat([token_row(wl, t, attempts[t]) for t in range(m)])


def attn_norm_weight(wl: Workload) -> torch.Tensor:
    """The attention seam's norm weight, bf16(1 + N(0, 0.1)) [H] on the host
    (its own stream; drawn like the FFN norm weight)."""
    return _bf16(1.0 + 0.1 * _rng(wl.seed, _TAG_ATTN_NORM).standard_normal(wl.dims.hidden))


def router_inputs(wl: Workload) -> dict:
    """norm_w bf16 [H], gate_w bf16 [E, H], bias f32 [E] on the host."""
    d = wl.dims
    norm_w = _bf16(1.0 + 0.1 * _rng(wl.seed, _TAG_NORM).standard_normal(d.hidden))
    gate_w = _bf16(0.02 * _rng(wl.seed, _TAG_GATE).standard_normal((d.experts, d.hidden)))
    r = _rng(wl.seed, _TAG_BIAS)
    if wl.bias == "normal":
        b = 0.01 * r.standard_normal(d.experts)
    elif wl.bias == "uniform":
        b = r.uniform(-0.01, 0.01, d.experts)
    elif wl.bias == "zipf":
        c = wl.extra.get("zipf_c", ZIPF_C)
        perm = _rng(wl.seed, _TAG_PERM).permutation(d.experts)
        b = np.zeros(d.experts)
        b[perm] = c * (np.arange(1, d.experts + 1, dtype=np.float64) ** -1.2)
    else:
        raise ValueError(wl.bias)
    return {"norm_w": norm_w, "gate_w": gate_w,
            "bias": torch.from_numpy(b.astype(np.float32))}


def _block_quant(w: torch.Tensor):
    """fp32 [R, C] -> (e4m3 bytes uint8 [R, C], codes uint8 [R/32, C/32]) with
    the synthesis rule of the module header."""
    r, c = w.shape
    blocks = w.view(r // 32, 32, c // 32, 32)
    amax = blocks.abs().amax(dim=(1, 3))
    _, e = torch.frexp(amax)  # amax = m * 2^e, m in [0.5, 1)
    e = e.to(torch.int32)
    code = (127 + e - 8).clamp(1, 254)
    # the multiplier 2^(127 - code) built from its fp32 bit pattern (exact)
    mul = ((254 - code) << 23).to(torch.int32).view(torch.float32)
    scaled = blocks * mul[:, None, :, None]
    b = scaled.view(r, c).to(torch.float8_e4m3fn).view(torch.uint8)
    return b, code.to(torch.uint8)


# E2M1 magnitudes in code order (codes 0..7) and the midpoints between them
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def _row_quant_fp4(w: torch.Tensor):
    """fp32 [R, C] -> (E2M1 pairs uint8 [R, C/2], codes uint8 [R, C/32]): per
    row and 32 columns a power-of-two scale 2^(e - 2) with 2^(e-1) <= amax <
    2^e (scaled magnitudes below 4), code 127 + e - 2, values rounded to the
    nearest E2M1 value (ties to the even code); element 2j in the low nibble
    of byte j. A synthesis rule for the inputs, like _block_quant."""
    r, c = w.shape
    blocks = w.view(r, c // 32, 32)
    amax = blocks.abs().amax(dim=2)
    _, e = torch.frexp(amax)
    code = (127 + e.to(torch.int32) - 2).clamp(1, 254)
    mul = ((254 - code) << 23).to(torch.int32).view(torch.float32)
    v = (blocks * mul[..., None]).view(r, c)
    a = v.abs()
    mid = torch.tensor(_E2M1_MID, dtype=a.dtype, device=a.device)
    k = torch.bucketize(a, mid)  # a <= mid[k] and a > mid[k - 1]
    tie = (k < len(_E2M1_MID)) & (a == mid[k.clamp(max=len(_E2M1_MID) - 1)]) & (k % 2 == 1)
    k = torch.where(tie, k + 1, k)
    nib = (k | (torch.signbit(v).to(k.dtype) << 3)).to(torch.uint8)
    packed = nib[:, 0::2] | (nib[:, 1::2] << 4)
    return packed.contiguous(), code.to(torch.uint8)


def _expert_gen(device, seed: int, tag: int, e: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tag * 65_537 + e) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def expert_weights(wl: Workload, device="cpu", experts=None, sigma: float = 0.02) -> dict:
    """Routed + shared expert weights on ``device``.

    Returns w13 uint8 [E, 2I, H], w13_s uint8 [E, 2I/32, H/32], w2 uint8
    [E, H, I], w2_s uint8 [E, H/32, I/32] (E2M1 routed experts: w13 [E, 2I,
    H/2], w13_s [E, 2I, H/32], w2 [E, H, I/2], w2_s [E, H, I/32]) and the
    shared expert's sw13 / sw13_s / sw2 / sw2_s (E4M3) without the E axis. ``experts``: optional iterable of routed
    expert ids to draw (others stay zero) -- each expert has its own stream, so
    a subset draws the same values as the whole.
    """
    d = wl.dims
    h, i, ish = d.hidden, d.inter, d.shared_inter
    dev = torch.device(device)
    fp4 = d.routed == "e2m1"
    if fp4:  # E2M1 pairs, one code per row per 32 columns
        w13 = torch.zeros(d.experts, 2 * i, h // 2, dtype=torch.uint8, device=dev)
        w13_s = torch.zeros(d.experts, 2 * i, h // 32, dtype=torch.uint8, device=dev)
        w2 = torch.zeros(d.experts, h, i // 2, dtype=torch.uint8, device=dev)
        w2_s = torch.zeros(d.experts, h, i // 32, dtype=torch.uint8, device=dev)
    else:
        w13 = torch.zeros(d.experts, 2 * i, h, dtype=torch.uint8, device=dev)
        w13_s = torch.zeros(d.experts, 2 * i // 32, h // 32, dtype=torch.uint8, device=dev)
        w2 = torch.zeros(d.experts, h, i, dtype=torch.uint8, device=dev)
        w2_s = torch.zeros(d.experts, h // 32, i // 32, dtype=torch.uint8, device=dev)
    quant = _row_quant_fp4 if fp4 else _block_quant
    todo = range(d.experts) if experts is None else sorted(set(int(e) for e in experts))
    for e in todo:
        g = _expert_gen(dev, wl.seed, _T_W13, e)
        w13[e], w13_s[e] = quant(torch.randn(2 * i, h, generator=g, device=dev) * sigma)
        g = _expert_gen(dev, wl.seed, _T_W2, e)
        w2[e], w2_s[e] = quant(torch.randn(h, i, generator=g, device=dev) * sigma)
    g = _expert_gen(dev, wl.seed, _T_SW13, 0)
    sw13, sw13_s = _block_quant(torch.randn(2 * ish, h, generator=g, device=dev) * sigma)
    g = _expert_gen(dev, wl.seed, _T_SW2, 0)
    sw2, sw2_s = _block_quant(torch.randn(h, ish, generator=g, device=dev) * sigma)
    return {"w13": w13, "w13_s": w13_s, "w2": w2, "w2_s": w2_s,
            "sw13": sw13, "sw13_s": sw13_s, "sw2": sw2, "sw2_s": sw2_s}


def algorithmic_bytes(dims: MoeDims, unique_routed: int) -> int:
    """Bytes one step must stream: gate weight + bias + the shared expert +
    the unique routed experts touched (weights and their E8M0 scales)."""
    return dims.router_bytes() + dims.shared_bytes() + unique_routed * dims.expert_bytes()


def algorithmic_flops(dims: MoeDims, m: int) -> int:
    """2 * 3 * I * H per (token, expert) over k routed + 1 shared expert."""
    return 2 * 3 * dims.inter * dims.hidden * m * (dims.topk + 1)
