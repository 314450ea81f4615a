"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bar (per workload): E4M3 bytes and E8M0 codes of the seam bit-exact (taken on
the GPU's own normed row, since the fp32 norm may differ from the float64
oracle by one bf16 ulp at a rounding boundary); normed within 1 bf16 ulp;
top-k expert ids bit-exact as ordered lists (inputs drawn with every top-k gap
> 1e-3); routing weights within 1e-5 relative of the oracle's router on the
same (GPU) normed rows; the bf16 output within a normwise relative error of
5e-3 of the oracle.
"""

import numpy as np
import pytest
import torch

from mxfp8_moe_decode_gb300 import workloads as W
from oracle import moe as O

from _harness import Layer, bf16_ulp_diff, f64, gapped_tokens, rel_err

pytestmark = pytest.mark.gpu

OUT_TOL = 5e-3
W_RTOL = 1e-5


def check(L: Layer, x: torch.Tensor, tokens=None, label=""):
    out, dbg = L.run(x)
    ref = L.oracle(x, tokens=tokens)
    m = x.shape[0]
    # seam
    ulp = bf16_ulp_diff(f64(dbg["normed"]), ref.normed)
    assert ulp.max() <= 1, (label, int(ulp.max()))
    xb, xc = O.seam_quant(f64(dbg["normed"]))
    assert np.array_equal(dbg["x8"].numpy(), xb), label
    assert np.array_equal(dbg["x8_codes"].numpy(), xc), label
    same = ulp.reshape(m, -1, 32).max(-1) == 0  # groups whose normed values agree
    assert np.array_equal(dbg["x8_codes"].numpy()[same], ref.codes[same]), label
    # router: ids against the oracle on its own rows (the inputs' top-k gaps
    # make them robust to a 1-ulp normed difference); weights and logits
    # against the oracle's router on the GPU's normed rows (the same input)
    assert np.array_equal(dbg["topk_ids"].numpy(), ref.routing.ids), label
    d = L.wl.dims
    rt = O.router(f64(dbg["normed"]), f64(L.ri["gate_w"]), f64(L.ri["bias"]), d.topk)
    assert np.array_equal(dbg["topk_ids"].numpy(), rt.ids), label
    np.testing.assert_allclose(dbg["topk_w"].numpy(), rt.weights, rtol=W_RTOL)
    np.testing.assert_allclose(dbg["logits"].numpy(), rt.logits, rtol=1e-4, atol=2e-5)
    # output
    rows = list(range(m)) if tokens is None else list(tokens)
    err = rel_err(f64(out)[rows], ref.out[rows])
    assert err <= OUT_TOL, (label, err)
    assert L.layer.status() == 0
    return err, int((ulp > 0).sum())


@pytest.fixture(scope="module")
def tiny():
    L = Layer(W.WORKLOADS["tiny_m1"])
    yield L
    L.close()


def test_tiny_m1(tiny):
    x, _ = gapped_tokens(tiny.wl, tiny.ri)
    err, nd = check(tiny, x, label="tiny_m1")
    print(f"tiny_m1: rel err {err:.2e}, normed ulp diffs {nd}")


@pytest.mark.parametrize("m", [2, 3, 7, 15, 16, 17, 31, 32, 33, 47, 48])
def test_tiny_ragged_m(tiny, m):
    # every MMA N (16 / 32 / 48) and ragged token counts per expert
    x, _ = gapped_tokens(tiny.wl, tiny.ri, m=m)
    err, _ = check(tiny, x, label=f"tiny m={m}")
    assert err <= OUT_TOL


def test_tiny_special_rows(tiny):
    # an all-zero row (codes 0, bytes 0) and tiny negatives next to large values
    # (bytes 0x80); the zero row's routing is decided by the bias alone
    x, _ = gapped_tokens(tiny.wl, tiny.ri, m=4)
    x[1] = 0
    x[2, ::7] = -1e-30
    out, dbg = tiny.run(x)
    ref = tiny.oracle(x)
    xb, xc = O.seam_quant(f64(dbg["normed"]))
    assert np.array_equal(dbg["x8"].numpy(), xb) and np.array_equal(dbg["x8_codes"].numpy(), xc)
    assert np.all(dbg["x8"].numpy()[1] == 0) and np.all(dbg["x8_codes"].numpy()[1] == 0)
    assert np.any(dbg["x8"].numpy()[2] == 0x80)
    assert np.array_equal(dbg["topk_ids"].numpy(), ref.routing.ids)
    rows = [0, 2, 3]
    assert rel_err(f64(out)[rows], ref.out[rows]) <= OUT_TOL
    assert np.all(np.isfinite(f64(out)))


@pytest.mark.parametrize("m", [3, 6])  # the seam fused into the router, and its own kernel
def test_tiny_nonfinite_rows_stay_in_their_rows(tiny, m):
    # A NaN row and a row with one infinite element: the choice keys are
    # integers made from the scores' bits and the expert index, so top-k
    # still picks k distinct valid experts for them, nothing reads or writes
    # out of bounds, and no error is raised. Every token's output depends on
    # its own row only, so the finite rows must still match the oracle run on
    # those rows alone.
    x, _ = gapped_tokens(tiny.wl, tiny.ri, m=m)
    x[1] = float("nan")
    x[m - 1, 5] = float("inf")
    out, dbg = tiny.run(x)
    assert tiny.layer.status() == 0
    d = tiny.wl.dims
    ids = dbg["topk_ids"].numpy()
    for r in (1, m - 1):
        assert len(set(ids[r].tolist())) == d.topk and ids[r].min() >= 0 and ids[r].max() < d.experts
    rows = [r for r in range(m) if r not in (1, m - 1)]
    ref = tiny.oracle(x[rows])
    assert np.array_equal(ids[rows], ref.routing.ids)
    assert rel_err(f64(out)[rows], ref.out) <= OUT_TOL
    assert np.all(np.isfinite(f64(out)[rows]))


def test_tiny_deterministic_and_graph(tiny):
    x, _ = gapped_tokens(tiny.wl, tiny.ri, m=5)
    xd = x.to(tiny.dev)
    a = tiny.layer.step(xd).clone()
    b = tiny.layer.step(xd).clone()
    assert torch.equal(a, b)
    s = torch.cuda.Stream(tiny.dev)
    out = torch.empty_like(xd)
    s.wait_stream(torch.cuda.current_stream(tiny.dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        tiny.layer.step(xd, out=out)  # warm-up on the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            tiny.layer.step(xd, out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, a)
    assert tiny.layer.status() == 0


def test_tiny_range_errors(tiny):
    from mxfp8_moe_decode_gb300._lib import MOE_ERR_RANGE, MoeError
    d = tiny.wl.dims
    for m in (0, d.max_tokens + 1):
        x = torch.zeros(m, d.hidden, dtype=torch.bfloat16, device=tiny.dev)
        with pytest.raises(MoeError) as ei:
            tiny.layer.step(x)
        assert ei.value.code == MOE_ERR_RANGE


@pytest.mark.parametrize("name,m", [("tiny_m1", 1), ("small_m4", 4), ("tiny_m1", 7)])
def test_unit_table(name, m):
    """The unit table the expert kernel derives from the per-expert row counts
    (written by its CTA 0) and the partial-output row of every pick the
    combine derives from the same counts (MOE_REGION_TOKPOS): routed experts
    with rows in increasing id, contiguous row runs from 0 in that order, the
    shared expert last with rows M k .. M k + M - 1; a pick's row lies in its
    expert's run and the picks of one expert fill the run exactly."""
    from mxfp8_moe_decode_gb300._lib import REGION_ACTIVE, REGION_TOKPOS
    L = Layer(W.WORKLOADS[name])
    try:
        d = L.wl.dims
        x, _ = gapped_tokens(L.wl, L.ri, m=m)
        _, dbg = L.run(x)
        ids = dbg["topk_ids"].numpy()
        K, E = d.topk, d.experts
        counts = np.bincount(ids.reshape(-1), minlength=E)
        active = np.nonzero(counts)[0]
        units = len(active) + 1
        assert L.layer.unique_experts() == len(active)
        act = L.layer.scratch_region(REGION_ACTIVE, torch.int32).numpy().reshape(-1, 4)[:units]
        first = np.concatenate([[0], np.cumsum(counts[active])])
        np.testing.assert_array_equal(act[:-1, 0], active)
        np.testing.assert_array_equal(act[:-1, 1], first[:-1])
        np.testing.assert_array_equal(act[:-1, 2], counts[active])
        assert tuple(act[-1, :3]) == (E, m * K, m)
        pos = L.layer.scratch_region(REGION_TOKPOS, torch.int32).numpy()[: m * (K + 1)]
        pos = pos.reshape(m, K + 1)
        np.testing.assert_array_equal(pos[:, K], m * K + np.arange(m))
        start = dict(zip(active.tolist(), first[:-1].tolist()))
        for e in active.tolist():
            rows = np.sort(pos[:, :K][ids == e])
            np.testing.assert_array_equal(rows, start[e] + np.arange(counts[e]))
    finally:
        L.close()


@pytest.mark.parametrize("m", [1, 2, 5, 16, 17, 33, 48])
def test_fp4_routed_experts(m):
    """MXFP4 routed experts (E2M1 weights, per-row 1 x 32 codes) against the
    oracle's per-row dequantisation, every MMA N bucket and ragged rows."""
    L = Layer(W.WORKLOADS["tiny_fp4"])
    try:
        x, _ = gapped_tokens(L.wl, L.ri, m=m)
        err, _ = check(L, x, label=f"tiny_fp4 m={m}")
        print(f"tiny_fp4 m={m}: rel err {err:.2e}")
    finally:
        L.close()


def test_fp4_every_code():
    """The synthesis rule never draws E2M1 code 7 (6.0): routed weights of
    uniformly random bytes (all 16 codes in both nibbles) with per-row codes
    spread over 2^-10 .. 2^-6, against the oracle's decoding."""
    def edit(ew):
        g = torch.Generator(device=ew["w13"].device).manual_seed(1234)
        for k in ("w13", "w2"):
            ew[k].copy_(torch.randint(0, 256, ew[k].shape, generator=g, device=ew[k].device,
                                      dtype=torch.int32).to(torch.uint8))
            ew[k + "_s"].copy_(torch.randint(117, 122, ew[k + "_s"].shape, generator=g,
                                             device=ew[k].device, dtype=torch.int32)
                               .to(torch.uint8))
    L = Layer(W.WORKLOADS["tiny_fp4"], edit_weights=edit)
    try:
        w = L.ew["w13"].cpu().numpy()
        assert len(np.unique(w & 15)) == 16 and len(np.unique(w >> 4)) == 16
        for m in (1, 17, 48):
            x, _ = gapped_tokens(L.wl, L.ri, m=m)
            err, _ = check(L, x, label=f"fp4 every code m={m}")
            print(f"fp4 every code m={m}: rel err {err:.2e}")
    finally:
        L.close()


def test_e4m3_every_code():
    """The synthesis rule keeps scaled weights below 256: routed and shared
    weights of uniformly random E4M3 bytes (every finite code, NaN bytes
    0x7F / 0xFF excluded) with block codes 113..117, against the oracle."""
    def edit(ew):
        g = torch.Generator(device=ew["w13"].device).manual_seed(4321)
        for k in ("w13", "w2", "sw13", "sw2"):
            b = torch.randint(0, 254, ew[k].shape, generator=g, device=ew[k].device,
                              dtype=torch.int32)
            b = torch.where(b >= 0x7F, b + 1, b)  # skip 0x7F; 0xFF is never drawn
            ew[k].copy_(b.to(torch.uint8))
            ew[k + "_s"].copy_(torch.randint(113, 118, ew[k + "_s"].shape, generator=g,
                                             device=ew[k].device, dtype=torch.int32)
                               .to(torch.uint8))
    L = Layer(W.WORKLOADS["tiny_m1"], edit_weights=edit)
    try:
        w = L.ew["w13"].cpu().numpy()
        assert len(np.unique(w)) == 254 and not np.any((w == 0x7F) | (w == 0xFF))
        for m in (1, 17, 48):
            x, _ = gapped_tokens(L.wl, L.ri, m=m)
            err, _ = check(L, x, label=f"e4m3 every code m={m}")
            print(f"e4m3 every code m={m}: rel err {err:.2e}")
    finally:
        L.close()


def test_step_launches(tiny):
    """Steps of at most 4 tokens run the seam inside the router: one launch fewer."""
    L = tiny.layer
    assert [L.step_launches(m) for m in (1, 4, 5, tiny.wl.dims.max_tokens)] == [4, 4, 5, 5]
    assert L.step_launches(0) == 0 and L.step_launches(tiny.wl.dims.max_tokens + 1) == 0


def test_small_m4():
    L = Layer(W.WORKLOADS["small_m4"])
    try:
        x, _ = gapped_tokens(L.wl, L.ri)
        err, nd = check(L, x, label="small_m4")
        print(f"small_m4: rel err {err:.2e}, normed ulp diffs {nd}")
    finally:
        L.close()


# every output row of every full-size workload against the oracle (which
# evaluates each touched expert once over all the rows that picked it)
@pytest.mark.parametrize("name,sample", [("full_m1", None), ("full_m16", None),
                                         ("full_m48_uniform", None),
                                         ("full_m48_zipf", None),
                                         ("full_e384_m1", None),
                                         ("full_e384_m48", None),
                                         ("full_e384_fp4_m1", None),
                                         ("full_e384_fp4_m48", None)])
def test_full_size(name, sample):
    L = Layer(W.WORKLOADS[name])
    try:
        x, _ = gapped_tokens(L.wl, L.ri)
        err, nd = check(L, x, tokens=sample, label=name)
        print(f"{name}: rel err {err:.2e} on tokens {sample}, normed ulp diffs {nd}, "
              f"unique routed experts {L.layer.unique_experts()}")
    finally:
        L.close()
        del L
        torch.cuda.empty_cache()


# ---------------------------------------------------------------- limits and degenerate routing

def test_max_experts_and_topk():
    # 512 routed experts (two per top-k thread, 16 candidate groups), top-16
    # (picks beyond one combine batch), 48 tokens
    wl = W.Workload("limits_e512_k16", W.MoeDims(256, 512, 16, 256, 256), 48, 5, "normal")
    # at H = 256 the scores of 512 experts crowd together; a bias with 0.05
    # steps over a seeded permutation spreads the choices so that draws with
    # every top-17 gap > 1e-3 exist
    perm = np.random.default_rng([5, 99]).permutation(512)
    bias = torch.zeros(512, dtype=torch.float32)
    bias[torch.from_numpy(perm)] = -0.05 * torch.arange(512, dtype=torch.float32)
    L = Layer(wl, bias=bias)
    try:
        x, _ = gapped_tokens(L.wl, L.ri)
        err, _ = check(L, x, label="E512 k16")
        print(f"E512 k16 M48: rel err {err:.2e}")
    finally:
        L.close()


def test_max_hidden_and_inter():
    # H = I = 8192: 64 K stages per w13 and w2 task, 128 w13 tiles per expert,
    # the largest seam row; output checked on token 0 (the oracle's expert path
    # at this size is slow), seam and routing on every token
    wl = W.Workload("limits_h8192_i8192", W.MoeDims(8192, 32, 2, 8192, 8192), 2, 6, "normal")
    L = Layer(wl)
    try:
        x, _ = gapped_tokens(L.wl, L.ri)
        err, _ = check(L, x, tokens=[0], label="H8192 I8192")
        print(f"H8192 I8192: rel err {err:.2e}")
    finally:
        L.close()


def test_fp4_limits():
    # MXFP4 routed experts at the largest widths (64 K stages per task, 4-bit
    # rows of 4 KB) and with 512 experts at top-16 and the smallest widths
    # (4-bit rows of 128 bytes: the copy's minimum box row)
    wl = W.Workload("limits_fp4_h8192", W.MoeDims(8192, 32, 2, 8192, 8192, routed="e2m1"), 2, 6,
                    "normal")
    L = Layer(wl)
    try:
        x, _ = gapped_tokens(L.wl, L.ri)
        err, _ = check(L, x, tokens=[0], label="fp4 H8192 I8192")
        print(f"fp4 H8192 I8192: rel err {err:.2e}")
    finally:
        L.close()
    wl = W.Workload("limits_fp4_e512", W.MoeDims(256, 512, 16, 256, 256, routed="e2m1"), 48, 5,
                    "normal")
    perm = np.random.default_rng([5, 99]).permutation(512)
    bias = torch.zeros(512, dtype=torch.float32)
    bias[torch.from_numpy(perm)] = -0.05 * torch.arange(512, dtype=torch.float32)
    L = Layer(wl, bias=bias)
    try:
        x, _ = gapped_tokens(L.wl, L.ri)
        err, _ = check(L, x, label="fp4 E512 k16")
        print(f"fp4 E512 k16 M48: rel err {err:.2e}")
    finally:
        L.close()


def test_every_token_on_the_same_experts():
    # a bias that sends all 48 tokens to the same k experts: every routed unit
    # has 48 rows (MMA N = 48), the other experts are idle
    wl = W.WORKLOADS["tiny_m1"]
    d = wl.dims
    bias = W.router_inputs(wl)["bias"].clone()
    hot = [5, 17, 33, 60]
    for j, e in enumerate(hot):
        bias[e] = 5.0 + 2.0 * j  # steps larger than any score difference
    L = Layer(wl, bias=bias)
    try:
        x, _ = gapped_tokens(L.wl, L.ri, m=48)
        err, _ = check(L, x, label="same experts")
        out, dbg = L.run(x)
        ids = dbg["topk_ids"].numpy()
        assert np.all(ids == np.array(hot[::-1])[None, :]), ids[:2]
        assert L.layer.unique_experts() == d.topk
        print(f"same experts M48: rel err {err:.2e}")
    finally:
        L.close()
