"""Pins of the oracle's norm, router, expert and combine (CPU only).

Checked against hand-worked values (tests/golden/rmsnorm_cases.txt,
tests/golden/expert_hand_case.txt), closed forms of silu / sigmoid, brute
force over every k-subset for the top-k, an independent per-element loop for
the expert contraction, the one-token / one-expert reduction of the whole
step, and token-permutation invariance.
"""

import itertools
import math
import os

import numpy as np
import pytest

from oracle import moe
from oracle.mx import dequant_rows, quant_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rms_cases():
    out = []
    with open(os.path.join(GOLDEN, "rmsnorm_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            x, w, eps, want = [p.strip() for p in line.split("|")]
            out.append((np.array(x.split(), float), np.array(w.split(), float),
                        float(eps), np.array(want.split(), float)))
    return out


def test_rmsnorm_hand_cases():
    cases = _rms_cases()
    assert len(cases) >= 5
    for x, w, eps, want in cases:
        got = moe.rmsnorm(x[None, :], w, eps)[0]
        assert np.array_equal(got, want), (x, w, got, want)


def test_attn_norm_closed_forms_and_ffn_rounding():
    # a constant row c: mean(x^2) = c^2, so y = c w / sqrt(c^2 + eps)
    w = np.linspace(0.5, 1.5, 64)
    y = moe.attn_norm(np.full((1, 64), 2.0), w, 0.0)[0]
    assert np.array_equal(y, w)
    y = moe.attn_norm(np.full((1, 64), -3.0), w, 1e-6)[0]
    assert np.allclose(y, -3.0 * w / math.sqrt(9.0 + 1e-6), rtol=1e-15, atol=0)
    # alternating +-a with unit weight: +-a / sqrt(a^2 + eps)
    x = np.tile([0.5, -0.5], 32)[None, :]
    y = moe.attn_norm(x, np.ones(64), 1e-6)[0]
    assert np.allclose(y, x[0] / math.sqrt(0.25 + 1e-6), rtol=1e-15, atol=0)
    # the FFN seam's norm is its bf16 rounding (hand-worked bf16 values)
    for x, w, eps, want in _rms_cases():
        got = moe.bf16_rne(moe.attn_norm(x[None, :], w, eps))[0]
        assert np.array_equal(got, want), (x, got, want)


def test_attn_seam_quant_hand_case():
    """fp32 values that bf16 cannot hold, quantised by hand (E4M3: bias 7,
    3 mantissa bits, subnormals k * 2^-9; codes from ceil(log2(amax / 448)))."""
    v = np.zeros(128)
    # group 0: amax 448 -> code 127, multiplier 1
    v[0:7] = [448.0, 1.0625, 1.0625 + 2.0 ** -20, 1.0 + 2.0 ** -20, -0.0, 2.0 ** -10,
              3.0 * 2.0 ** -10]
    # group 1: amax 897 -> 897 / 448 = 2.0022 -> code 129, multiplier 1/4
    v[32:35] = [897.0, 896.0, -1.0]
    # group 2: all zero -> code 0
    # group 3: amax 448 (1 + 2^-20) (bf16 would round it to 448, code 127) -> code 128
    v[96:98] = [448.0 * (1.0 + 2.0 ** -20), 1.0]
    b, c = moe.attn_seam_quant(v[None, :])
    assert list(c[0]) == [127, 129, 0, 128]
    want = np.zeros(128, dtype=np.uint8)
    # 448 = 1.75 * 2^8 -> 0 1111 110; 1.0625 ties 1.0 / 1.125 -> even 1.0 (0x38);
    # just above the tie -> 1.125 (0x39); 1 + 2^-20 -> 1.0; -0.0 keeps its sign;
    # 2^-10 ties 0 / 2^-9 -> 0; 1.5 * 2^-9 ties 2^-9 / 2^-8 -> 2^-8 (0x02)
    want[0:7] = [0x7E, 0x38, 0x39, 0x38, 0x80, 0x00, 0x02]
    # 897/4 = 224.25 -> 224 = 1.75 * 2^7 (0 1110 110); 896/4 = 224; -1/4 = -(0 0101 000)
    want[32:35] = [0x76, 0x76, 0xA8]
    # 448 (1 + 2^-20) / 2 -> 224; 1/2 = 2^-1 -> 0 0110 000
    want[96:98] = [0x76, 0x30]
    assert np.array_equal(b[0], want), [hex(x) for x in b[0][:8]]
    with pytest.raises(ValueError):
        moe.attn_seam_quant(np.full((1, 32), 0.1))  # 0.1 is not an fp32 value


def test_silu_sigmoid_closed_forms():
    assert moe.sigmoid(0.0) == 0.5
    assert math.isclose(moe.silu(1.0), 0.7310585786300049, rel_tol=1e-15)
    assert math.isclose(moe.silu(-1.0), -0.2689414213699951, rel_tol=1e-15)
    assert moe.silu(0.0) == 0.0
    assert math.isclose(moe.silu(2.0), 1.7615941559557646, rel_tol=1e-15)
    assert abs(moe.silu(-40.0)) < 1e-15


def test_topk_bruteforce():
    rng = np.random.default_rng(11)
    for trial in range(200):
        e = int(rng.integers(2, 11))
        k = int(rng.integers(1, e + 1))
        c = rng.standard_normal(e)
        ids = moe.topk_desc(c[None], k)[0]
        # the unique k-subset whose every member beats every non-member
        best = [s for s in itertools.combinations(range(e), k)
                if min(c[list(s)]) > max(np.delete(c, list(s)), default=-np.inf)]
        assert len(best) == 1
        assert sorted(ids.tolist()) == sorted(best[0])
        assert all(c[ids[j]] > c[ids[j + 1]] for j in range(k - 1))


def test_topk_ties_lower_index_first():
    c = np.array([[1.0, 2.0, 2.0, 0.0, 2.0]])
    assert moe.topk_desc(c, 2)[0].tolist() == [1, 2]
    assert moe.topk_desc(c, 4)[0].tolist() == [1, 2, 4, 0]


def test_router_hand_case():
    normed = np.array([[1.0, 0.0]])
    gate_w = np.array([[0.0, 5.0], [2.0, 1.0], [-1.0, 0.0], [1.0, -3.0]])
    bias = np.zeros(4)
    rt = moe.router(normed, gate_w, bias, 2)
    assert rt.logits.tolist() == [[0.0, 2.0, -1.0, 1.0]]
    assert rt.ids.tolist() == [[1, 3]]
    s1, s3 = 0.8807970779778823, 0.7310585786300049  # sigmoid(2), sigmoid(1)
    assert np.allclose(rt.weights, [[s1 / (s1 + s3), s3 / (s1 + s3)]], rtol=1e-15)
    # the bias moves the choice but not the weights (scores stay unbiased)
    rt = moe.router(normed, gate_w, np.array([0.0, 0.0, 0.5, 0.0]), 2)
    assert rt.ids.tolist() == [[1, 2]]
    s2 = 0.2689414213699951  # sigmoid(-1)
    assert np.allclose(rt.weights, [[s1 / (s1 + s2), s2 / (s1 + s2)]], rtol=1e-15)


def _hand_expert():
    h = 32
    w13 = np.zeros((64, h), np.uint8)
    w13[:32, 0] = 0x38
    w13[32 + np.arange(32), np.arange(32)] = 0x38
    w13_s = np.array([[128], [127]], np.uint8)
    w2 = np.zeros((h, 32), np.uint8)
    w2[np.arange(32), np.arange(32)] = 0x38
    w2_s = np.array([[127]], np.uint8)
    return w13, w13_s, w2, w2_s


def _golden_expert():
    vals = {}
    with open(os.path.join(GOLDEN, "expert_hand_case.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float.fromhex(v) if v.startswith("0x") else float(v)
    return vals


def test_expert_hand_case():
    g = _golden_expert()
    ew = moe.ExpertWeights.from_quantised(*_hand_expert())
    x_hat = dequant_rows(np.full((1, 32), 0x38, np.uint8), np.array([[127]], np.uint8))
    y, h, hb, hc = moe.expert(x_hat, ew)
    assert np.allclose(h, g["h"], rtol=1e-15)
    assert np.all(hc == int(g["h8_code"])) and np.all(hb == int(g["h8_byte"]))
    assert np.all(y == g["y"])


def test_expert_matches_elementwise_loop():
    # the vectorised expert against a plain triple loop over the dequantised
    # values, on random small shapes (independent arithmetic path)
    rng = np.random.default_rng(3)
    h, inter = 64, 64
    w13b = rng.integers(0, 0x7E, (2 * inter, h)).astype(np.uint8) | (rng.integers(0, 2, (2 * inter, h)) << 7).astype(np.uint8)
    w13s = rng.integers(115, 125, (2 * inter // 32, h // 32)).astype(np.uint8)
    w2b = rng.integers(0, 0x7E, (h, inter)).astype(np.uint8)
    w2s = rng.integers(110, 120, (h // 32, inter // 32)).astype(np.uint8)
    ew = moe.ExpertWeights.from_quantised(w13b, w13s, w2b, w2s)
    x8, xc = quant_rows(rng.standard_normal((1, h)))
    x_hat = dequant_rows(x8, xc)
    y, hh, hb, hc = moe.expert(x_hat, ew)
    from oracle.numerics import e4m3_decode
    gu = np.zeros(2 * inter)
    for r in range(2 * inter):
        acc = 0.0
        for c in range(h):
            wv = float(e4m3_decode(w13b[r, c])) * 2.0 ** (int(w13s[r // 32, c // 32]) - 127)
            xv = float(e4m3_decode(x8[0, c])) * 2.0 ** (int(xc[0, c // 32]) - 127)
            acc += wv * xv
        gu[r] = acc
    href = [gu[i] / (1 + math.exp(-gu[i])) * gu[inter + i] for i in range(inter)]
    assert np.allclose(hh[0], href, rtol=1e-12, atol=1e-300)
    hq = dequant_rows(hb, hc)[0]
    yref = np.zeros(h)
    for r in range(h):
        yref[r] = sum(float(e4m3_decode(w2b[r, c])) * 2.0 ** (int(w2s[r // 32, c // 32]) - 127) * hq[c]
                      for c in range(inter))
    assert np.allclose(y[0], yref, rtol=1e-12)


def _tiny_layer(rng, h=64, e=8, inter=64):
    def q(shape, code_lo, code_hi):
        b = rng.integers(0, 0x7E, shape).astype(np.uint8) | (rng.integers(0, 2, shape) << 7).astype(np.uint8)
        s = rng.integers(code_lo, code_hi, (shape[0] // 32, shape[1] // 32)).astype(np.uint8)
        return b, s
    experts = [moe.ExpertWeights.from_quantised(*q((2 * inter, h), 112, 118), *q((h, inter), 112, 118))
               for _ in range(e)]
    shared = moe.ExpertWeights.from_quantised(*q((2 * inter, h), 112, 118), *q((h, inter), 112, 118))
    norm_w = 1 + 0.1 * rng.standard_normal(h)
    gate_w = 0.1 * rng.standard_normal((e, h))
    bias = 0.01 * rng.standard_normal(e)
    return experts, shared, norm_w, gate_w, bias


def test_one_token_one_expert_reduction():
    # k = 1 and a shared expert whose output is zero: out = bf16(y_e) with
    # weight exactly 1, whatever expert the router picks
    rng = np.random.default_rng(4)
    experts, shared, norm_w, gate_w, bias = _tiny_layer(rng)
    zero = moe.ExpertWeights(w13=shared.w13, w2=np.zeros_like(shared.w2))
    x = moe.bf16_rne(rng.standard_normal((1, 64)))
    res = moe.decode_step(x, norm_w, gate_w, bias, 1, lambda e: experts[e], lambda: zero)
    e = int(res.routing.ids[0, 0])
    assert res.routing.weights[0, 0] == 1.0
    y = moe.expert(dequant_rows(res.x8, res.codes), experts[e])[0]
    assert np.array_equal(res.out, moe.bf16_rne(y))


def test_identical_routed_experts_sum_once():
    # every routed expert the same: whatever the router picks, the k picks'
    # normalised weights sum to 1, so out = bf16(y_routed + y_shared); a
    # dropped pick, an unnormalised weight or a shared term added twice fails
    rng = np.random.default_rng(12)
    experts, shared, norm_w, gate_w, bias = _tiny_layer(rng)
    same = experts[0]
    x = moe.bf16_rne(rng.standard_normal((3, 64)))
    for k in (1, 2, 3):
        res = moe.decode_step(x, norm_w, gate_w, bias, k, lambda e: same, lambda: shared)
        assert np.allclose(res.routing.weights.sum(axis=1), 1.0, rtol=0, atol=1e-15)
        xh = dequant_rows(res.x8, res.codes)
        y = moe.expert(xh, same)[0]
        ysh = moe.expert(xh, shared)[0]
        # the weights sum to 1 only up to rounding: compare before the bf16 step
        acc = np.einsum("mk,mh->mh", res.routing.weights, y) + ysh
        want = moe.bf16_rne(acc)
        assert np.array_equal(res.out, want), k
        assert np.allclose(acc, y + ysh, rtol=1e-14, atol=1e-14)


def test_step_token_permutation_invariance():
    rng = np.random.default_rng(9)
    experts, shared, norm_w, gate_w, bias = _tiny_layer(rng)
    x = moe.bf16_rne(rng.standard_normal((5, 64)))
    perm = np.array([3, 0, 4, 1, 2])
    a = moe.decode_step(x, norm_w, gate_w, bias, 2, lambda e: experts[e], lambda: shared)
    b = moe.decode_step(x[perm], norm_w, gate_w, bias, 2, lambda e: experts[e], lambda: shared)
    assert np.array_equal(a.out[perm], b.out)
    assert np.array_equal(a.x8[perm], b.x8)
    assert np.array_equal(a.routing.ids[perm], b.routing.ids)


def test_step_token_subset_matches_full():
    rng = np.random.default_rng(10)
    experts, shared, norm_w, gate_w, bias = _tiny_layer(rng)
    x = moe.bf16_rne(rng.standard_normal((4, 64)))
    full = moe.decode_step(x, norm_w, gate_w, bias, 2, lambda e: experts[e], lambda: shared)
    part = moe.decode_step(x, norm_w, gate_w, bias, 2, lambda e: experts[e], lambda: shared,
                           tokens=[2])
    assert np.array_equal(full.out[2], part.out[2])
    assert np.all(np.isnan(part.out[[0, 1, 3]]))


def test_topk_gaps_hand_rows():
    # the smallest gap among the k + 1 largest choices; the rows are shuffled
    # too (the function must sort them first)
    k = 3
    rows = np.array([
        [0.9, 0.6, 0.3, 0.0, -0.3],        # clean: every gap is 0.3
        [0.9, 0.5, 0.4995, 0.1, 0.0],      # a close pair inside the top k (picks 2 and 3)
        [0.9, 0.6, 0.3, 0.2995, 0.0],      # a close pair at the boundary (pick k vs k + 1)
        [0.9, 0.6, 0.3, 0.0, -0.0004],     # a close pair below the k + 1 largest: ignored
        [0.9, 0.6, 0.6, 0.0, -0.3],        # a tie inside the top k: gap 0
    ])
    want = np.array([0.3, 0.0005, 0.0005, 0.3, 0.0])
    np.testing.assert_allclose(moe.topk_gaps(rows, k), want, rtol=0, atol=1e-12)
    perm = [3, 0, 4, 2, 1]
    np.testing.assert_allclose(moe.topk_gaps(rows[:, perm], k), want, rtol=0, atol=1e-12)
    # k = 1: only the gap between the largest and the second largest counts
    np.testing.assert_allclose(moe.topk_gaps(rows, 1), [0.3, 0.4, 0.3, 0.3, 0.3],
                               rtol=0, atol=1e-12)


def test_combine_hand_two_tokens():
    # token 0: picks output 1 and 3 with weights 0.25, 0.75 and the shared
    # expert 0.5: 0.25 + 2.25 + 0.5 = 3.0; token 1 the picks swapped:
    # 0.75 + 0.75 + 0.5 = 2.0; token 2: 0.5 * 1 + 0.5 * 5 + 2^-7 = 3 + 2^-7
    # lies halfway between the bf16 neighbours 3 and 3 + 2^-6 and rounds to
    # the even one, 3.0
    h = 4
    y = np.zeros((3, 2, h))
    y[0, 0], y[0, 1] = 1.0, 3.0
    y[1, 0], y[1, 1] = 3.0, 1.0
    y[2, 0], y[2, 1] = 1.0, 5.0
    w = np.array([[0.25, 0.75], [0.25, 0.75], [0.5, 0.5]])
    ysh = np.array([[0.5] * h, [0.5] * h, [2.0 ** -7] * h])
    out = moe.combine(y, w, ysh)
    assert np.array_equal(out, np.array([[3.0] * h, [2.0] * h, [3.0] * h]))


def _const_expert(y_byte: int, y_code: int) -> moe.ExpertWeights:
    """H = I = 32 expert whose output is a constant on the all-ones x_hat row:
    gate rows 1.0 * 2^1 -> g = 32 * 2 = 64 and silu(64) = 64 in float64; up
    rows 1.0 * 2^-11 -> u = 2^-6, so h = 1 (code 119, byte 0x78, exact); the
    w2 entries are y_byte * 2^(y_code - 127), so y = 32 * that value."""
    w13 = np.full((64, 32), 0x38, np.uint8)            # E4M3 1.0
    w13_s = np.array([[128], [116]], np.uint8)         # gate block x2, up block x2^-11
    w2 = np.full((32, 32), y_byte, np.uint8)
    w2_s = np.array([[y_code]], np.uint8)
    return moe.ExpertWeights.from_quantised(w13, w13_s, w2, w2_s)


def test_step_pairs_weights_with_their_picks():
    # normed = 1 (x = 1, w = 1, eps = 0), so the logits are the gate rows'
    # sums: 0, ln 3, -ln 3, 0 -> scores 1/2, 3/4, 1/4, 1/2; the bias makes the
    # choices -0.5, 0.75, 0.85, -0.5, so k = 2 picks [2, 1] with weights
    # 1/4 and 3/4. Expert 1 outputs 1 (0x38 * 2^-5 * 32), expert 2 outputs 3
    # (0x3C = 1.5, * 2^-4 * 32), the shared expert 0.5 (0x38 * 2^-6 * 32), the
    # unpicked ones 32: out = 1/4 * 3 + 3/4 * 1 + 1/2 = 2. Pairing weight j
    # with another pick gives 3; the mirror case (the two outputs swapped)
    # gives 3 where a wrong pairing gives 2.
    h = 32
    ln3 = math.log(3.0)
    gate_w = np.zeros((4, h))
    gate_w[1] = ln3 / h
    gate_w[2] = -ln3 / h
    bias = np.array([-1.0, 0.0, 0.6, -1.0])
    x = np.ones((1, h))
    other = _const_expert(0x38, 127)
    one, three = _const_expert(0x38, 122), _const_expert(0x3C, 123)
    half = _const_expert(0x38, 121)
    for e1, e2, want in ((one, three, 2.0), (three, one, 3.0)):
        experts = {0: other, 1: e1, 2: e2, 3: other}
        res = moe.decode_step(x, np.ones(h), gate_w, bias, 2, lambda e: experts[e],
                              lambda: half, eps=0.0)
        assert np.array_equal(res.normed, np.ones((1, h)))
        assert res.routing.ids.tolist() == [[2, 1]]
        np.testing.assert_allclose(res.routing.weights, [[0.25, 0.75]], rtol=1e-14)
        assert np.array_equal(res.out, np.full((1, h), want)), (want, res.out[0, :4])
