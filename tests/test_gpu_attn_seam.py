"""GPU parity of the attention-seam MXFP8 (moe_attn_seam_x8) against the oracle.

Bar: the fp32 norm outputs within 1e-5 relative of the float64 oracle (the
fp32 sum of squares has at most 8 * 8 chained roundings per owner plus 7 in
the reduction tree, about 4.2e-6 relative at H = 8192, halved by the inverse
square root; rsqrtf's 2 ulps and the products' 3 roundings add < 4e-7); the
E4M3 bytes and E8M0 codes bit-exact against the oracle's quant of the GPU's
own fp32 norm outputs.
"""

import numpy as np
import pytest
import torch

from mxfp8_moe_decode_gb300 import attn_seam_x8
from mxfp8_moe_decode_gb300 import workloads as W
from oracle import moe as O

pytestmark = pytest.mark.gpu

YS_RTOL = 1e-5


def _f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def _check(x, w, eps=1e-6, label=""):
    dev = torch.device("cuda:0")
    xd, wd = x.to(dev), w.to(dev)
    M, H = x.shape
    ys = torch.empty((M, H), dtype=torch.float32, device=dev)
    x8, codes, _ = attn_seam_x8(xd, wd, eps, ys=ys)
    torch.cuda.synchronize()
    ref = O.attn_norm(_f64(x), _f64(w), eps)
    got = _f64(ys)
    scale = np.abs(ref).max(axis=-1, keepdims=True)
    err = np.abs(got - ref) / np.maximum(scale, 1e-300)
    assert err.max() <= YS_RTOL, (label, float(err.max()))
    b, c = O.attn_seam_quant(got)
    assert np.array_equal(x8.cpu().numpy(), b), label
    assert np.array_equal(codes.cpu().numpy(), c), label
    # without ys the kernel gives the same bytes
    x8b, codesb, none = attn_seam_x8(xd, wd, eps)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(x8b, x8) and torch.equal(codesb, codes), label
    return float(err.max())


@pytest.mark.parametrize("name", ["tiny_m1", "full_m48_uniform"])
@pytest.mark.parametrize("m", [1, 4, 7, 48])
def test_attn_seam_workload_rows(name, m):
    wl = W.WORKLOADS[name]
    x = W.token_rows(wl, m=m)
    err = _check(x, W.attn_norm_weight(wl), label=f"{name} m={m}")
    print(f"{name} m={m}: ys max rel err {err:.2e}")


def test_attn_seam_special_rows():
    # an all-zero row (codes 0, bytes 0), tiny negatives beside large values
    # (bytes 0x80), a row of large values, and a single nonzero column
    H = 1024
    g = torch.Generator().manual_seed(7)
    x = torch.randn(4, H, generator=g)
    x[0] = 0.0
    x[1, ::32] = 200.0
    x[1, 1::32] = -1e-7
    x[2] *= 3e4
    x[3] = 0.0
    x[3, 5] = -2.5
    x = x.to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    _check(x, w, label="special")


@pytest.mark.parametrize("H", [32, 96, 8192])
def test_attn_seam_widths(H):
    # the narrowest row (one group; most owners idle), a width that is not a
    # multiple of 128, and the widest row
    g = torch.Generator().manual_seed(H)
    x = torch.randn(5, H, generator=g).to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    _check(x, w, eps=1e-5, label=f"H={H}")


def test_attn_seam_rejects_bad_shapes():
    dev = torch.device("cuda:0")
    x = torch.zeros(49, 256, dtype=torch.bfloat16, device=dev)
    w = torch.ones(256, dtype=torch.bfloat16, device=dev)
    from mxfp8_moe_decode_gb300._lib import MoeError
    with pytest.raises(MoeError):
        attn_seam_x8(x, w)  # M = 49
    with pytest.raises(ValueError):
        attn_seam_x8(x[:4, :250].contiguous(), w[:250].contiguous())  # H % 32
