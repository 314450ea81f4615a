"""Pins of the oracle's E8M0 code and 32-group quantisation (CPU only).

The code formula is the device page's ``mx_code``: clamp(ceil(log2(amax/448))
+ 127, 0, 254), amax floored at FLT_MIN. Checked against hand-worked cases
(tests/golden/mx_code_cases.txt), against exact rational arithmetic for every
positive finite bf16 amax, and against the closed form 127 + k at every
power-of-two multiple 448 * 2^k.
"""

import os
from fractions import Fraction

import numpy as np
import pytest

from oracle.mx import (block_scale_shape, dequant_rows, dequant_weight, mx_code,
                       quant_rows)
from oracle.numerics import e4m3_decode

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    out = []
    with open(os.path.join(GOLDEN, "mx_code_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            out.append((float.fromhex(parts[1]), int(parts[2])))
    return out


def test_mx_code_hand_cases():
    cases = _cases()
    assert len(cases) >= 8
    for amax, code in cases:
        assert int(mx_code(amax)) == code, (amax, code)


def test_mx_code_powers_of_two():
    # 448 * 2^k is exact in fp32 for k in [-134, 119]; the code is 127 + k
    # (clamped at 0), and just above the boundary it is one more.
    for k in range(-134, 120):
        a = np.float32(448.0) * np.float32(2.0) ** k if k > -126 else np.ldexp(np.float32(1.75), k + 8)
        a = np.float32(a)
        assert float(a) == 448.0 * 2.0 ** k
        assert int(mx_code(float(a))) == max(127 + k, 0), k
        if 127 + k >= 1 and k < 119:
            above = np.nextafter(a, np.float32(np.inf))
            assert int(mx_code(float(above))) == 128 + k, k


def _exact_code(a: Fraction) -> int:
    """clamp(ceil(log2(a / 448)) + 127, 0, 254) in exact rationals (a > 0)."""
    q = a / 448
    e = 0
    # smallest e with 2^e >= q
    if q >= 1:
        while Fraction(2) ** e < q:
            e += 1
    else:
        while Fraction(2) ** (e - 1) >= q:
            e -= 1
    return min(max(e + 127, 0), 254)


def test_mx_code_all_bf16_vs_exact():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)  # positive finite bf16 patterns
    vals = (bits << 16).view(np.float32).astype(np.float64)
    got = mx_code(vals)
    flt_min = Fraction(1, 2 ** 126)
    for v, c in zip(vals[::7], got[::7]):  # every 7th value: ~4700 exact checks
        a = max(Fraction(float(v)), flt_min)
        assert int(c) == _exact_code(a), v
    # the whole set is monotone non-decreasing in amax
    assert np.all(np.diff(got.astype(np.int64)) >= 0)


def test_quant_rows_cases():
    # group with amax 448: code 127, bytes are the E4M3 of the values themselves
    v = np.zeros((1, 32))
    v[0, :4] = [448.0, -1.0, 0.5, 3.0]
    b, c = quant_rows(v)
    assert c.tolist() == [[127]]
    assert b[0, :4].tolist() == [0x7E, 0xB8, 0x30, 0x44]
    assert np.all(b[0, 4:] == 0)
    # all-zero group: code 0, bytes 0
    b, c = quant_rows(np.zeros((2, 64)))
    assert np.all(c == 0) and np.all(b == 0)
    # a tiny negative next to a large value rounds to -0 (0x80)
    v = np.zeros((1, 32))
    v[0, 0] = 1.0
    v[0, 1] = -1e-9
    b, c = quant_rows(v)
    assert int(c[0, 0]) == 119 and b[0, 1] == 0x80
    # scaling by 2^(127 - code) is exact: 1.0 at code 119 becomes 256 -> 0x78
    assert b[0, 0] == 0x78


def test_quant_dequant_error_bound():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((64, 256)).astype(np.float32).astype(np.float64)
    b, c = quant_rows(v)
    r = dequant_rows(b, c)
    g = v.reshape(64, 8, 32)
    amax = np.abs(g).max(-1, keepdims=True)
    # E4M3 has 3 mantissa bits: relative error <= 2^-4 of the value for normal
    # codes, plus the subnormal quantum 2^-9 * scale; scale <= amax / 224
    err = np.abs(r.reshape(64, 8, 32) - g)
    scale = amax / 224.0
    assert np.all(err <= np.abs(g) * 2.0 ** -4 + scale * 2.0 ** -10 + 1e-300)


def test_block_scale_layout():
    # runner page: wqkv [1792, 5120] e4m3 with a [56, 160] E8M0 scale
    assert block_scale_shape(1792, 5120) == (56, 160)
    assert block_scale_shape(4096, 5120) == (128, 160)  # full-size w13
    assert block_scale_shape(5120, 2048) == (160, 64)  # full-size w2
    with pytest.raises(ValueError):
        block_scale_shape(100, 64)


def test_dequant_weight_block_addressing():
    w = np.zeros((96, 64), dtype=np.uint8)
    codes = np.full((3, 2), 127, dtype=np.uint8)
    w[33, 40] = 0x38  # 1.0, in block (1, 1)
    codes[1, 1] = 130  # scale 2^3
    w[70, 5] = 0xC0  # -2.0, in block (2, 0)
    codes[2, 0] = 120  # scale 2^-7
    d = dequant_weight(w, codes)
    assert d[33, 40] == 8.0
    assert d[70, 5] == -2.0 * 2.0 ** -7
    assert np.count_nonzero(d) == 2
    with pytest.raises(ValueError):
        dequant_weight(w, codes[:2])
    assert e4m3_decode(np.uint8(0xC0)) == -2.0


def test_dequant_fp4_rows_per_row_scales():
    """Each row's 32-column block has its own code (1 x 32 scales): an
    independent element loop over a hand-set pattern."""
    from oracle.mx import dequant_fp4_rows
    R, C = 3, 64
    rng = np.random.default_rng(5)
    packed = rng.integers(0, 256, size=(R, C // 2), dtype=np.uint8)
    code = np.array([[127, 130], [120, 127], [0, 254]], dtype=np.uint8)
    got = dequant_fp4_rows(packed, code)
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for r in range(R):
        for c in range(C):
            byte = int(packed[r, c // 2])
            nib = byte & 0xF if c % 2 == 0 else byte >> 4
            v = table[nib & 7] * (-1.0 if nib & 8 else 1.0)
            want = v * 2.0 ** (int(code[r, c // 32]) - 127)
            assert got[r, c] == want, (r, c, got[r, c], want)
    with pytest.raises(ValueError):
        dequant_fp4_rows(packed, code[:, :1])


def test_fp4_synthesis_rule():
    """The input generator's MXFP4 weights (workloads._row_quant_fp4), decoded
    by the oracle: each value within half an E2M1 spacing of its draw (a
    quarter-spacing of the scale below 2, a half above), ties to the even code,
    codes 127 + e - 2 for 2^(e-1) <= amax < 2^e."""
    import torch
    from mxfp8_moe_decode_gb300 import workloads as W
    from oracle.mx import dequant_fp4_rows
    g = torch.Generator().manual_seed(3)
    w = torch.randn(16, 256, generator=g) * 0.02
    w[0, :32] = 0.0
    w[1, :8] = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, -1.25, 3.9]) * 2.0 ** -6
    p, c = W._row_quant_fp4(w)
    assert p.shape == (16, 128) and c.shape == (16, 8)
    got = dequant_fp4_rows(p.numpy(), c.numpy())
    v = w.double().numpy()
    scale = np.repeat(2.0 ** (c.numpy().astype(np.int64) - 127), 32, axis=1)
    q = v / scale
    spacing = np.where(np.abs(q) < 2, 0.5, 1.0)
    assert np.all(np.abs(got / scale - q) <= spacing / 2 + 1e-12)
    amax = np.abs(v.reshape(16, 8, 32)).max(axis=2)
    nz = amax > 0
    e = np.floor(np.log2(amax[nz])) + 1
    assert np.array_equal(c.numpy()[nz].astype(np.int64), (127 + e - 2).astype(np.int64))
    # the hand-set ties (amax 3.9 * 2^-6 -> scale 2^-6): to the even code
    assert got[1, :8].tolist() == [x * 2.0 ** -6 for x in (0.0, 1.0, 1.0, 2.0, 2.0, 4.0, -1.0, 4.0)]
