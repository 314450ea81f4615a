"""Shared helpers of the GPU parity tests: seeded inputs with a top-k gap
(redrawing rows through the oracle's router), the layer on the GPU, and the
oracle's expert accessors over the same weight tensors."""

from __future__ import annotations

import numpy as np
import torch

from mxfp8_moe_decode_gb300 import MoeDecode
from mxfp8_moe_decode_gb300 import workloads as W
from oracle import moe as O

GAP = 1e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().double().cpu().numpy()


def gapped_tokens(wl: W.Workload, ri: dict, m: int | None = None, max_attempts: int = 200):
    """Token rows whose choice values have every top-(k+1) gap > 1e-3 (oracle
    router, float64). Returns (x bf16 [m, H] host, attempts per row)."""
    m = wl.tokens if m is None else m
    d = wl.dims
    nw, gw, b = f64(ri["norm_w"]), f64(ri["gate_w"]), f64(ri["bias"])
    attempts = [0] * m
    for t in range(m):
        while True:
            row = W.token_row(wl, t, attempts[t])
            normed = O.rmsnorm(f64(row), nw, d.eps)
            rt = O.router(normed, gw, b, d.topk)
            if O.topk_gaps(rt.choice, d.topk)[0] > GAP:
                break
            attempts[t] += 1
            if attempts[t] >= max_attempts:
                raise RuntimeError(f"no gapped draw for row {t}")
    return W.token_rows(wl, attempts=attempts, m=m), attempts


class Layer:
    """The workload's layer on the GPU plus oracle accessors over the same
    weight tensors (copied to the host one expert at a time)."""

    def __init__(self, wl: W.Workload, device="cuda:0", max_tokens: int | None = None,
                 bias: torch.Tensor | None = None, edit_weights=None):
        self.wl = wl
        d = wl.dims
        self.dev = torch.device(device)
        self.ri = W.router_inputs(wl)
        if bias is not None:  # a routing scenario the workload's bias does not give
            self.ri["bias"] = bias.to(torch.float32).cpu()
        self.ew = W.expert_weights(wl, device=self.dev)
        if edit_weights is not None:  # a weight pattern the synthesis rule does not give
            edit_weights(self.ew)
        weights = {"norm_w": self.ri["norm_w"].to(self.dev), "gate_w": self.ri["gate_w"].to(self.dev),
                   "bias": self.ri["bias"].to(self.dev), **self.ew}
        self.layer = MoeDecode(d.hidden, d.experts, d.topk, d.inter, weights,
                               max_tokens=max_tokens or d.max_tokens, eps=d.eps,
                               routed=d.routed)
        self._cache: dict = {}

    def expert(self, e: int) -> O.ExpertWeights:
        if e not in self._cache:
            ew = self.ew
            make = (O.ExpertWeights.from_fp4 if self.wl.dims.routed == "e2m1"
                    else O.ExpertWeights.from_quantised)
            self._cache[e] = make(
                ew["w13"][e].cpu().numpy(), ew["w13_s"][e].cpu().numpy(),
                ew["w2"][e].cpu().numpy(), ew["w2_s"][e].cpu().numpy())
        return self._cache[e]

    def shared(self) -> O.ExpertWeights:
        if "sh" not in self._cache:
            ew = self.ew
            self._cache["sh"] = O.ExpertWeights.from_quantised(
                ew["sw13"].cpu().numpy(), ew["sw13_s"].cpu().numpy(),
                ew["sw2"].cpu().numpy(), ew["sw2_s"].cpu().numpy())
        return self._cache["sh"]

    def run(self, x: torch.Tensor):
        """One GPU step with every debug output; returns (out, debug) on the host."""
        xd = x.to(self.dev)
        dbg = self.layer.debug_buffers(x.shape[0])
        out = self.layer.step(xd, debug=dbg)
        torch.cuda.synchronize(self.dev)
        return out.cpu(), {k: v.cpu() for k, v in dbg.items()}

    def oracle(self, x: torch.Tensor, tokens=None) -> O.StepResult:
        d = self.wl.dims
        return O.decode_step(f64(x), f64(self.ri["norm_w"]), f64(self.ri["gate_w"]),
                             f64(self.ri["bias"]), d.topk, self.expert, self.shared, d.eps,
                             tokens=tokens)

    def close(self):
        self.layer.close()


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in units of bf16 ulps (both arrays hold bf16 values)."""
    ia = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64)
    ib = torch.from_numpy(b.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64)
    # map sign-magnitude to a monotone integer line
    ia = np.where(ia < 0, -(ia & 0x7FFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFF), ib)
    return np.abs(ia - ib)
