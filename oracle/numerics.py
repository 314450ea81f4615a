"""Rounding and the E4M3 codec, written from their definitions.

TEST INFRASTRUCTURE ONLY (see the package header).

* ``bf16_rne``: round a float64 to the nearest bfloat16 (8 significant bits,
  fp32 exponent range, ties to even), in one step from float64. Used for the
  bf16 MoE input row ("store_normed", layer page) and the bf16 layer output
  (``out [M, HIDDEN] bf16``, runner page, ``DSV41MonoLayer._outs``).
* ``fp32_rn``: IEEE single rounding (numpy's float32 cast / arithmetic).
* E4M3 (OCP FP8 E4M3FN): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
  bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no
  infinity; largest finite 448 (the pages' FP8_MAX in ``mx_code``, device
  page). ``e4m3_decode`` builds the value of every byte from that definition;
  ``e4m3_encode_rne`` rounds to the nearest representable value, ties to the
  even mantissa, as ``fp8_pack4`` ("Four f32 (in range) -> ... E4M3 bytes,
  RNE", device page) does. Inputs to the encoder are in range (|v| <= 448):
  the method clamps before it converts (``clamp_fp8`` in ``store_x8``, layer
  page).

* E2M1 (OCP MX FP4): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa
  bit; exponent field 0 is subnormal (m/2); no infinity or NaN; values 0,
  0.5, 1, 1.5, 2, 3, 4, 6 and their negatives. The runner page's routed
  weights are ``torch.float4_e2m1fn_x2`` (two per byte): element 2j sits in
  the low nibble of byte j (``unpack_fp4x2``).

Pins (tests/test_oracle_numerics.py): all 256 decoded values against torch's
float8_e4m3fn and hand values from the OCP definition; every representable
value encodes to itself; every midpoint goes to the even neighbour and one
ulp either side goes to the nearer one; 10^6 random values against torch's
float8_e4m3fn cast; bf16_rne against torch's bfloat16 cast of fp32 values and
hand-worked ties.
"""

from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0


def fp32_rn(v):
    """IEEE binary32 round-to-nearest-even of float64 value(s)."""
    return np.asarray(v, dtype=np.float64).astype(np.float32)


def bf16_rne(v):
    """Round float64 value(s) to the nearest bfloat16 value, ties to even.

    One rounding straight from float64 (no fp32 step): the quantum is
    2^(e - 8) for |v| in [2^(e-1), 2^e), floored at the subnormal quantum
    2^-133. Returns float64 holding bf16-exact values.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    nz = v != 0
    _, e = np.frexp(v[nz])
    e = np.maximum(e, -125)  # bf16 normal exponents reach 2^-126 = 0.5 * 2^-125
    quantum = np.ldexp(1.0, e - 8)
    out[nz] = np.rint(v[nz] / quantum) * quantum  # np.rint rounds half to even
    # keep the sign of zero results (e.g. -tiny -> -0.0)
    out = np.where(np.signbit(v) & (out == 0), -0.0, out)
    return out


def _e4m3_value(byte: int) -> float:
    """Value of one E4M3 byte from the OCP FP8 E4M3FN definition."""
    s = -1.0 if byte & 0x80 else 1.0
    exp = (byte >> 3) & 0xF
    man = byte & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:
        return s * (man / 8.0) * 2.0 ** -6
    return s * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


E4M3_VALUES = np.array([_e4m3_value(b) for b in range(256)], dtype=np.float64)

# Non-negative finite codes 0x00..0x7E in increasing value order (the bit
# pattern order of a sign-magnitude float is its value order).
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = E4M3_VALUES[:0x7F]


def e4m3_decode(codes):
    """E4M3 bytes -> float64 values (NaN for 0x7F / 0xFF)."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode_rne(v):
    """float64 value(s) with |v| <= 448 -> E4M3 bytes, round to nearest even.

    The sign bit is kept for values that round to zero (-tiny -> 0x80).
    """
    v = np.asarray(v, dtype=np.float64)
    if np.any(np.isnan(v)) or np.any(np.abs(v) > E4M3_MAX):
        raise ValueError("e4m3_encode_rne: input outside [-448, 448]")
    a = np.abs(v)
    # hi = first representable value >= a; lo = the one below it
    hi = np.searchsorted(_POS_VALUES, a, side="left")
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    vhi = _POS_VALUES[hi]
    vlo = _POS_VALUES[lo]
    exact = vhi == a
    d_lo = a - vlo
    d_hi = vhi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((_POS_CODES[hi] & 1) == 0))
    code = np.where(exact, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    sign = np.signbit(v).astype(np.uint8) << 7
    return (code | sign).astype(np.uint8)


def _e2m1_value(nibble: int) -> float:
    """Value of one E2M1 code (4 bits) from the OCP MX FP4 definition."""
    s = -1.0 if nibble & 0x8 else 1.0
    exp = (nibble >> 1) & 0x3
    man = nibble & 0x1
    if exp == 0:
        return s * (man / 2.0)
    return s * (1.0 + man / 2.0) * 2.0 ** (exp - 1)


E2M1_VALUES = np.array([_e2m1_value(n) for n in range(16)], dtype=np.float64)


def unpack_fp4x2(packed):
    """uint8 [..., C/2] holding two E2M1 codes per byte -> codes uint8 [..., C]
    (element 2j = the low nibble of byte j, element 2j + 1 = the high nibble)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def e2m1_decode(codes):
    """E2M1 codes (uint8 values 0..15) -> float64 values."""
    c = np.asarray(codes, dtype=np.uint8)
    if np.any(c > 15):
        raise ValueError("e2m1_decode: codes are 4-bit")
    return E2M1_VALUES[c]
