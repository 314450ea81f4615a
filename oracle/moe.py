"""The MoE decode step (FFN half), step by step, in float64.

TEST INFRASTRUCTURE ONLY (see the package header).

Inputs are numpy arrays holding exact values: bf16 tensors as float64 arrays
of their values, E4M3 tensors as uint8 bytes, E8M0 scales as uint8 codes,
f32 tensors as float64 arrays of their values.

Steps and the passages they follow:

1. ``rmsnorm`` -- the FFN seam's norm (``seam.stage_norm``, called in
   ``run_ffn``, layer page; its body is not on the pages) followed by
   ``store_normed`` ("the FFN seam's norm output -> the MoE input row (bf16)",
   layer page). Reading: normed = bf16(x * (mean(x^2) + eps)^(-1/2) * w), the
   weight taken as given, eps 1e-6.
2. ``seam_quant`` -- MXFP8 of the bf16 normed row in 32-groups (``store_x8``,
   layer page; ``mx_code``, device page), via :func:`oracle.mx.quant_rows`.
3. ``router`` -- logits = normed . gate_w^T (``gate_w [E, 5120] bf16``,
   runner page, ``MonoLayerWeights``); scores s = sigmoid(logit); selection on
   s + bias (``bias [E] f32 (e_score_correction_bias)``, same class); the k
   largest, ties to the lower expert index; weights s_j / sum_j s_j.
4. ``expert`` -- one expert on one token: gu = x_hat . W13_hat^T with both
   operands dequantised per 32 along K (``mfma_scaled``: block-scaled MMA with
   one E8M0 per 32-K block per operand, device page); rows [0, I) of w13 are
   the gate, rows [I, 2I) the up projection (``sgu`` "shared gate_up
   [2 inter, 5120]", runner page); h = silu(g) * u; h requantised per 32 along
   I from its fp32 value (as ``store_x8`` quantises f32 values, layer page);
   y = h_hat . W2_hat^T (``sw2`` "shared down [5120, inter]", runner page).
5. ``combine`` -- out = bf16(sum_j w_j * y_{id_j} + y_shared) (``out [M, HIDDEN]
   bf16``, ``DSV41MonoLayer._outs``, runner page). The residual is not added.

Outside the FFN step, the attention seam's input quant (``store_x8``, layer
page: "the attention seam's norm output ... -> vLLM's MXFP8 of each 32"):
``attn_norm`` is the same norm with the attention norm weight, not rounded
(``seam.stage_norm``'s outputs are f32), and ``attn_seam_quant`` quantises
those fp32 values in 32-groups with the same code and E4M3 rule.

Pins (tests/test_oracle_moe.py): hand-worked RMSNorm values
(tests/golden/rmsnorm_cases.txt), silu closed forms, brute-force top-k over
all k-subsets on small E, hand rows for ``topk_gaps`` (a close pair inside
the top k, a close pair at the k / k+1 boundary, a close pair below it that
must not count), an expert built from hand-chosen bytes and codes whose
result is worked out by hand, a hand ``combine`` on two tokens with unequal
weights, and, for the composed step, a hand-built layer whose two picked
experts output different constants with unequal weights (and its mirror, the
constants swapped), which fixes the pairing of weight j with pick j; plus
three invariants: the one-token / one-expert reduction, identical routed
experts (the picks' weights sum to one: out = bf16(y + y_shared) whatever is
picked) and token-permutation invariance. The composed step has no worked
example on the pages: beyond what those pins and invariants fix, its
end-to-end numbers on random layers are "parity unpinned".
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .mx import dequant_fp4_rows, dequant_rows, dequant_weight, quant_rows
from .numerics import bf16_rne, fp32_rn


def rmsnorm(x, w, eps: float = 1e-6):
    """normed = bf16_RNE(x * (mean_h(x^2) + eps)^(-1/2) * w), float64 math.

    x: float64 [M, H] (bf16 values), w: float64 [H] (bf16 values).
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return bf16_rne(x * r * w)


def seam_quant(normed):
    """MXFP8 of the bf16 normed rows: (x8 bytes [M, H], codes [M, H/32])."""
    return quant_rows(normed)


def attn_norm(x, w, eps: float = 1e-6):
    """The attention seam's norm output x * (mean_h(x^2) + eps)^(-1/2) * w in
    float64, not rounded (the GPU's fp32 values are compared to it within the
    fp32 error bound; its MXFP8 is taken on the GPU's own fp32 values).

    x: float64 [M, H] (bf16 values), w: float64 [H] (bf16 values).
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * w


def attn_seam_quant(ys):
    """MXFP8 of fp32 norm outputs (fp32-exact float64 [M, H]) in 32-groups:
    (x8 bytes [M, H], codes [M, H/32]) -- ``store_x8`` on the attention seam."""
    ys = np.asarray(ys, dtype=np.float64)
    if not np.array_equal(fp32_rn(ys), ys):
        raise ValueError("attn_seam_quant: the inputs must be fp32 values")
    return quant_rows(ys)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))


def topk_desc(c, k: int):
    """Indices of the k largest entries of each row of c, in decreasing order;
    equal values go to the lower index first."""
    c = np.asarray(c, dtype=np.float64)
    out = np.empty(c.shape[:-1] + (k,), dtype=np.int64)
    for idx in np.ndindex(*c.shape[:-1]):
        row = c[idx]
        order = np.lexsort((np.arange(row.shape[0]), -row))  # last key is primary
        out[idx] = order[:k]
    return out


@dataclass
class Routing:
    logits: np.ndarray  # float64 [M, E]
    scores: np.ndarray  # float64 [M, E], sigmoid(logits)
    choice: np.ndarray  # float64 [M, E], scores + bias
    ids: np.ndarray  # int64 [M, k], decreasing choice
    weights: np.ndarray  # float64 [M, k], normalised scores of ids


def router(normed, gate_w, bias, k: int) -> Routing:
    """Gate GEMV, sigmoid, bias-adjusted top-k, normalised weights."""
    logits = np.asarray(normed, dtype=np.float64) @ np.asarray(gate_w, dtype=np.float64).T
    s = sigmoid(logits)
    c = s + np.asarray(bias, dtype=np.float64)[None, :]
    ids = topk_desc(c, k)
    sel = np.take_along_axis(s, ids, axis=-1)
    wts = sel / np.sum(sel, axis=-1, keepdims=True)
    return Routing(logits=logits, scores=s, choice=c, ids=ids, weights=wts)


def topk_gaps(choice, k: int):
    """Per row: the smallest gap between consecutive entries among the k+1
    largest choice values (decides both which experts are picked and their
    order)."""
    c = -np.sort(-np.asarray(choice, dtype=np.float64), axis=-1)[..., : k + 1]
    return np.min(c[..., :-1] - c[..., 1:], axis=-1)


def silu(g):
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


@dataclass
class ExpertWeights:
    """One expert, dequantised: W13 [2I, H] (gate rows then up rows), W2 [H, I]."""

    w13: np.ndarray
    w2: np.ndarray

    @staticmethod
    def from_quantised(w13_b, w13_s, w2_b, w2_s) -> "ExpertWeights":
        return ExpertWeights(w13=dequant_weight(w13_b, w13_s), w2=dequant_weight(w2_b, w2_s))

    @staticmethod
    def from_fp4(w13_p, w13_s, w2_p, w2_s) -> "ExpertWeights":
        """MXFP4 routed expert (runner page: ``w13 [E, 2 inter, 2560] fp4x2``,
        ``w2 [E, 5120, inter / 2] fp4x2``, scales per row per 32 columns)."""
        return ExpertWeights(w13=dequant_fp4_rows(w13_p, w13_s), w2=dequant_fp4_rows(w2_p, w2_s))


def expert(x_hat, ew: ExpertWeights):
    """One expert on rows x_hat (float64 [n, H], dequantised MXFP8 activations).

    Returns (y float64 [n, H], h float64 [n, I] before requant,
    h8 bytes [n, I], h8 codes [n, I/32]).
    """
    inter = ew.w2.shape[1]
    gu = np.asarray(x_hat, dtype=np.float64) @ ew.w13.T
    g, u = gu[:, :inter], gu[:, inter:]
    h = silu(g) * u
    h32 = fp32_rn(h).astype(np.float64)
    hb, hc = quant_rows(h32)
    y = dequant_rows(hb, hc) @ ew.w2.T
    return y, h, hb, hc


def combine(y_routed, weights, y_shared):
    """out = bf16(sum_j weights[:, j] * y_routed[:, j] + y_shared).

    y_routed float64 [M, k, H], weights [M, k], y_shared [M, H].
    """
    acc = np.einsum("mk,mkh->mh", np.asarray(weights, dtype=np.float64), y_routed)
    return bf16_rne(acc + y_shared)


@dataclass
class StepResult:
    normed: np.ndarray
    x8: np.ndarray
    codes: np.ndarray
    routing: Routing
    out: np.ndarray


def decode_step(x, norm_w, gate_w, bias, topk: int, get_expert, get_shared,
                eps: float = 1e-6, tokens=None) -> StepResult:
    """The whole FFN half for rows x (float64 [M, H] bf16 values).

    get_expert(e) -> ExpertWeights of routed expert e; get_shared() -> the
    shared expert's. Only the experts some token picked are requested, each
    once. ``tokens``: optional subset of row indices whose output to compute
    (the seam and the router still run on every row); other rows of ``out``
    are NaN.
    """
    normed = rmsnorm(x, norm_w, eps)
    x8, codes = seam_quant(normed)
    rt = router(normed, gate_w, bias, topk)
    x_hat = dequant_rows(x8, codes)
    m, hdim = normed.shape
    rows = list(range(m)) if tokens is None else list(tokens)
    out = np.full((m, hdim), np.nan)
    if rows:
        y_routed = np.zeros((m, topk, hdim))
        wanted = sorted({int(e) for t in rows for e in rt.ids[t]})
        for e in wanted:
            # every (token, pick) that chose expert e, in one call: each output
            # row of ``expert`` depends on its own input row only (per-row
            # contraction, per-row requant along I)
            picks = [(t, j) for t in rows for j in range(topk) if rt.ids[t, j] == e]
            y = expert(x_hat[[t for t, _ in picks]], get_expert(e))[0]
            for (t, j), y_tj in zip(picks, y):
                y_routed[t, j] = y_tj
        y_shared = expert(x_hat[rows], get_shared())[0]
        out[rows] = combine(y_routed[rows], rt.weights[rows], y_shared)
    return StepResult(normed=normed, x8=x8, codes=codes, routing=rt, out=out)
