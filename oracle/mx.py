"""MXFP8: the E8M0 scale code of a 32-group and E4M3 quantisation with it.

TEST INFRASTRUCTURE ONLY (see the package header).

Source passages:

* ``mx_code`` (device page): the scale code of a 32-group is
  clamp(ceil(log2(amax / 448)) + 127, 0, 254) with amax floored at FLT_MIN;
  the pages take the quotient as an IEEE single division (``div_rn``:
  "x / d rounded to nearest (IEEE)") and its ceiling exponent from the bits
  (``ceil_exp``: "biased exponent of the smallest power of two >= v").
* ``mx_mul`` / ``rcp_pow2`` (device page): the quant multiplier 2^(127 - code).
* ``store_x8`` (layer page): amax over the 32 values of a group, the code,
  ``clamp_fp8(y * mul)`` then ``fp8_pack4`` (E4M3, RNE) -- one code byte per
  32 columns at ``t * X_GROUPS + col // 32`` (row-major [rows, cols/32]).
* ``fp8x8_bf16`` (device page): dequantisation = byte value x power-of-two
  scale, exact.
* ``MonoLayerWeights.check`` / ``AttnWeights.check`` (runner page): a weight
  [R, C] e4m3 has a [R/32, C/32] uint8 E8M0 scale, one code per 32 x 32 block
  (e.g. wqkv [1792, 5120] with a [56, 160] scale).
* ``MonoLayerWeights`` (runner page): the routed w13 / w2 are
  ``float4_e2m1fn_x2`` ([E, 2 inter, 2560] for 5120 columns) with scales of
  HIDDEN // 32 columns per weight row (``w13_s [E * 2 inter, HIDDEN // 32]``):
  one code per row per 32 columns (``dequant_fp4_rows``). The pages store
  them in AITER's shuffled orders; the plain row-major order is taken here.

Readings (where the pages leave a step open):

* The quotient q = fp32_RN(max(amax, FLT_MIN) / 448) follows ``div_rn``; the
  code is then clamp(ceil(log2 q) + 127, 0, 254) taken exactly on that fp32 q.
  For a normal q this is ``ceil_exp``'s bit rule. ``ceil_exp`` is stated for
  normal v only; for a subnormal q (amax < 448 * 2^-126) the formula itself is
  applied: code 1 for q in (2^-127, 2^-126), else 0. An all-zero group
  therefore gets code 0 and bytes 0x00.
* ``clamp_fp8`` clamps to [-448, 448] before the RNE convert.
* A value that rounds to zero keeps its sign (byte 0x80 for -tiny).

Pins (tests/test_oracle_mx.py): hand cases (448 -> 127, 448 * 2^k -> 127 + k,
just above -> 128 + k, 0 -> 0), every positive finite bf16 amax against the
exact rational ceil(log2(amax / 448)) via ``fractions.Fraction``, the
[1792, 5120] -> [56, 160] scale shape, a one-element block round trip, and the
golden cases in tests/golden/mx_code_cases.txt; ``dequant_fp4_rows`` by an
independent element loop with per-row codes (E2M1 itself is pinned in
tests/test_oracle_numerics.py against tests/golden/e2m1_values.txt).
"""

from __future__ import annotations

import numpy as np

from .numerics import E4M3_MAX, e2m1_decode, e4m3_decode, e4m3_encode_rne, unpack_fp4x2

FLT_MIN = 2.0 ** -126
GROUP = 32


def mx_code(amax) -> np.ndarray:
    """E8M0 code(s) of 32-group absolute maxima (fp32-exact inputs, >= 0)."""
    amax = np.asarray(amax, dtype=np.float64)
    a = np.maximum(amax, FLT_MIN).astype(np.float32)
    q = a / np.float32(E4M3_MAX)  # IEEE single division, round to nearest
    # ceil(log2 q) exactly: q = f * 2^e with f in [0.5, 1) (frexp of the fp32
    # value widened to float64, which is exact also for a subnormal q)
    f, e = np.frexp(q.astype(np.float64))
    c = np.where(f == 0.5, e - 1, e).astype(np.int64) + 127
    return np.clip(c, 0, 254).astype(np.uint8)


def mx_mul(code):
    """2^(127 - code): the quant multiplier of a code (float64, exact)."""
    return np.ldexp(1.0, 127 - np.asarray(code, dtype=np.int64))


def mx_scale(code):
    """2^(code - 127): the dequant scale of a code (float64, exact)."""
    return np.ldexp(1.0, np.asarray(code, dtype=np.int64) - 127)


def quant_rows(v):
    """Quantise rows of fp32-exact values in 32-groups along the last axis.

    v: float64 [..., K] with K % 32 == 0 -> (bytes uint8 [..., K],
    codes uint8 [..., K/32]).
    """
    v = np.asarray(v, dtype=np.float64)
    k = v.shape[-1]
    if k % GROUP:
        raise ValueError("quant_rows: last axis must be a multiple of 32")
    g = v.reshape(v.shape[:-1] + (k // GROUP, GROUP))
    amax = np.max(np.abs(g), axis=-1)
    code = mx_code(amax)
    y = g * mx_mul(code)[..., None]
    y = np.clip(y, -E4M3_MAX, E4M3_MAX)
    # np.clip keeps -0.0; the encoder keeps the sign of a zero result
    b = e4m3_encode_rne(y).reshape(v.shape)
    return b, code


def dequant_rows(b, code):
    """Inverse of quant_rows' encoding: bytes [..., K], codes [..., K/32] -> float64."""
    vals = e4m3_decode(b)
    k = vals.shape[-1]
    s = np.repeat(mx_scale(code), GROUP, axis=-1)
    if s.shape[-1] != k:
        raise ValueError("dequant_rows: codes do not cover the row")
    return vals * s


def block_scale_shape(rows: int, cols: int) -> tuple[int, int]:
    """Shape of the E8M0 scale of an [rows, cols] weight in 32 x 32 blocks."""
    if rows % GROUP or cols % GROUP:
        raise ValueError("block_scale_shape: dims must be multiples of 32")
    return rows // GROUP, cols // GROUP


def dequant_weight(b, code):
    """E4M3 weight [R, C] with a 32 x 32-block code [R/32, C/32] -> float64 [R, C].

    Element (r, c) is scaled by the code of block (r // 32, c // 32).
    """
    b = np.asarray(b)
    code = np.asarray(code)
    if code.shape != block_scale_shape(*b.shape):
        raise ValueError(f"dequant_weight: scale {code.shape} does not match {b.shape}")
    s = mx_scale(code)
    s = np.repeat(np.repeat(s, GROUP, axis=0), GROUP, axis=1)
    return e4m3_decode(b) * s


def dequant_fp4_rows(packed, code):
    """MXFP4 weight: E2M1 pairs [R, C/2] (``unpack_fp4x2`` order) with one code
    per row per 32 columns [R, C/32] -> float64 [R, C].

    Element (r, c) is scaled by code (r, c // 32): the runner page's routed
    w13 / w2 carry their scales per row ("per-row 1 x 32": ``w13_s`` has
    HIDDEN // 32 columns per weight row).
    """
    vals = e2m1_decode(unpack_fp4x2(packed))
    code = np.asarray(code)
    if code.shape != (vals.shape[0], vals.shape[1] // GROUP) or vals.shape[1] % GROUP:
        raise ValueError(f"dequant_fp4_rows: scale {code.shape} does not match {vals.shape}")
    return vals * np.repeat(mx_scale(code), GROUP, axis=1)
