"""Pins of the oracle's rounding and E4M3 codec (CPU only).

Each test checks the oracle against something other than itself: the OCP
E4M3 definition worked by hand (tests/golden/e4m3_values.txt), torch's own
float8_e4m3fn / bfloat16 casts (library routines), or properties that any
correct round-to-nearest-even must have.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle.numerics import (E4M3_VALUES, bf16_rne, e2m1_decode, e4m3_decode, e4m3_encode_rne,
                             unpack_fp4x2)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_e4m3():
    out = []
    with open(os.path.join(GOLDEN, "e4m3_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            b, v = line.split()[:2]
            out.append((int(b, 16), float(v)))
    return out


def test_e4m3_hand_values():
    cases = _golden_e4m3()
    assert len(cases) >= 15
    for b, v in cases:
        got = e4m3_decode(np.uint8(b))
        if math.isnan(v):
            assert math.isnan(got)
        else:
            assert got == v and math.copysign(1, got) == math.copysign(1, v), hex(b)


def test_e4m3_table_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(E4M3_VALUES))
    assert np.array_equal(ref[~nan], E4M3_VALUES[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(E4M3_VALUES[~nan]))
    assert nan.sum() == 2  # only S.1111.111


def test_e4m3_encode_identity():
    codes = np.array([b for b in range(256) if b not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3_decode(codes)
    assert np.array_equal(e4m3_encode_rne(vals), codes)


def test_e4m3_midpoints_go_to_even():
    pos = np.arange(0x7F)
    v = E4M3_VALUES[pos]
    mids = (v[:-1] + v[1:]) / 2
    got = e4m3_encode_rne(mids)
    want = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:]).astype(np.uint8)
    assert np.array_equal(got, want)
    # just either side of the midpoint goes to the nearer neighbour
    lo = np.nextafter(mids, -np.inf)
    hi = np.nextafter(mids, np.inf)
    assert np.array_equal(e4m3_encode_rne(lo), pos[:-1].astype(np.uint8))
    assert np.array_equal(e4m3_encode_rne(hi), pos[1:].astype(np.uint8))
    # negative side mirrors with the sign bit
    assert np.array_equal(e4m3_encode_rne(-mids), want | 0x80)


def test_e4m3_boundaries():
    assert e4m3_encode_rne(2.0 ** -10) == 0x00  # tie between 0 and 2^-9 -> even (0)
    assert e4m3_encode_rne(-(2.0 ** -10)) == 0x80
    assert e4m3_encode_rne(3 * 2.0 ** -10) == 0x02  # tie between 1 and 2 (x 2^-9) -> 2
    assert e4m3_encode_rne(-1e-30) == 0x80  # sign kept on a zero result
    assert e4m3_encode_rne(0.0) == 0x00
    assert e4m3_encode_rne(-0.0) == 0x80
    assert e4m3_encode_rne(2.0 ** -6) == 0x08  # smallest normal
    assert e4m3_encode_rne(448.0) == 0x7E
    assert e4m3_encode_rne(432.0) == 0x7E  # tie 416 | 448 -> 448 (even mantissa 6)
    assert e4m3_encode_rne(400.0) == 0x7C  # tie 384 | 416 -> 384 (even mantissa 4)
    with pytest.raises(ValueError):
        e4m3_encode_rne(449.0)


def test_e4m3_random_vs_torch():
    rng = np.random.default_rng(123)
    n = 1_000_000
    mag = np.exp2(rng.uniform(-14, 8.8, n)).astype(np.float32)
    v = (mag * rng.choice([-1, 1], n)).astype(np.float32)
    v = np.clip(v, -448, 448)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3_encode_rne(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rne_vs_torch():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) < 3e38)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = bf16_rne(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rne_hand_ties():
    assert bf16_rne(1 + 2.0 ** -8) == 1.0  # tie -> even
    assert bf16_rne(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    # one rounding from float64: 1 + 2^-8 + 2^-30 lies above the bf16 tie, but
    # an fp32 step first would land on the tie and then round down to 1.0
    assert bf16_rne(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7
    assert bf16_rne(-(1 + 2.0 ** -8 + 2.0 ** -30)) == -(1 + 2.0 ** -7)
    assert bf16_rne(2.0 ** -133) == 2.0 ** -133  # smallest bf16 subnormal
    assert bf16_rne(2.0 ** -134) == 0.0  # tie with zero -> even (zero)


def test_e2m1_hand_values():
    rows = []
    with open(os.path.join(GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                p = line.split()
                rows.append((int(p[0], 16), float(p[4])))
    assert [c for c, _ in rows] == list(range(16))
    got = e2m1_decode(np.arange(16, dtype=np.uint8))
    for c, v in rows:
        assert got[c] == v and math.copysign(1.0, got[c]) == math.copysign(1.0, v), (c, got[c], v)
    with pytest.raises(ValueError):
        e2m1_decode(np.uint8(16))


def test_fp4x2_nibble_order():
    # byte j holds element 2j in its low nibble and 2j + 1 in its high nibble
    p = np.array([[0x21, 0xF7, 0x80]], dtype=np.uint8)
    assert unpack_fp4x2(p).tolist() == [[0x1, 0x2, 0x7, 0xF, 0x0, 0x8]]
    assert e2m1_decode(unpack_fp4x2(p)).tolist() == [[0.5, 1.0, 6.0, -6.0, 0.0, -0.0]]
