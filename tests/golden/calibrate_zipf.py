"""Choose the Zipf(s=1.2) router-bias scale C of the 48-row full-size workload.

The workload wants 48 token rows to concentrate on about 32 hot experts. With
bias[perm[r]] = C * (r + 1)^-1.2, this script routes the workload's 48 rows
(first draw of every row) with the oracle's router and prints the smallest C
on a 1e-3 grid (up to 20) for which the rows touch between 28 and 36 distinct experts,
aiming at 32. The printed value is stored as ``ZIPF_C`` in
mxfp8_moe_decode_gb300/workloads.py.

Run: python tests/golden/calibrate_zipf.py
"""

import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))

from mxfp8_moe_decode_gb300 import workloads as W  # noqa: E402
from oracle import moe  # noqa: E402


def main():
    wl = W.WORKLOADS["full_m48_zipf"]
    d = wl.dims
    ri = W.router_inputs(wl)
    x = W.token_rows(wl).float().double().numpy()
    normed = moe.rmsnorm(x, ri["norm_w"].double().numpy(), d.eps)
    s = moe.sigmoid(normed @ ri["gate_w"].double().numpy().T)
    perm = W._rng(wl.seed, W._TAG_PERM).permutation(d.experts)
    shape = np.zeros(d.experts)
    shape[perm] = np.arange(1, d.experts + 1, dtype=np.float64) ** -1.2
    best = None
    for i in range(0, 20001):
        c = i * 1e-3
        bias = (c * shape).astype(np.float32).astype(np.float64)
        ids = moe.topk_desc(s + bias, d.topk)
        u = len(np.unique(ids))
        if 28 <= u <= 36 and (best is None or abs(u - 32) < abs(best[1] - 32)):
            best = (c, u)
            if u <= 32:
                break
    print(f"ZIPF_C = {best[0]:.3f}  (unique experts at M=48: {best[1]})")


if __name__ == "__main__":
    main()
