"""The device-side timeout path, made to run out in the allowed form: a
host-set toggle (moe_test_withhold_ready) keeps one unit's w13 tiles from
ever being reported done, so the w2 tasks of that unit wait on a flag that
nothing sets until their bounded wait (1 s) expires. No memory fault, no trap,
no endless loop: the kernel records MOE_ERR_TIMEOUT, lets its copies and MMAs
in flight complete, frees its tensor memory and returns; the stream
completes, the host reads the status, clears it, and the next step is
bit-identical to a clean one."""

import time

import pytest
import torch

from mxfp8_moe_decode_gb300 import workloads as W
from mxfp8_moe_decode_gb300._lib import MOE_ERR_TIMEOUT, MOE_OK

from _harness import Layer, gapped_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    L = Layer(W.WORKLOADS["tiny_m1"])
    yield L
    L.layer.test_withhold_ready(-1)
    L.close()


# unit 0 is the shared expert (in every step); units >= 1 are routed experts.
# M = 1 also runs the split w2 tiles (K-halves), M = 48 every MMA width.
@pytest.mark.parametrize("unit,m", [(0, 5), (1, 1), (2, 48)])
def test_timeout_reported_then_clean_step(tiny, unit, m):
    L = tiny.layer
    x, _ = gapped_tokens(tiny.wl, tiny.ri, m=m)
    xd = x.to(tiny.dev)
    clean = L.step(xd).clone()
    torch.cuda.synchronize(tiny.dev)
    assert L.status() == MOE_OK

    L.test_withhold_ready(unit)
    t0 = time.monotonic()
    L.step(xd)
    torch.cuda.current_stream(tiny.dev).synchronize()  # the kernels return
    waited = time.monotonic() - t0
    L.test_withhold_ready(-1)
    assert L.status() == MOE_ERR_TIMEOUT
    # one bounded wait (1 s) per CTA that took one of the unit's w2 tasks,
    # all at the same time, plus the teardown
    assert 0.9 < waited < 20.0, waited

    assert L.clear_status() == MOE_OK
    assert L.status() == MOE_OK
    again = L.step(xd).clone()
    torch.cuda.synchronize(tiny.dev)
    assert L.status() == MOE_OK
    assert torch.equal(again, clean)


def test_withhold_range(tiny):
    from mxfp8_moe_decode_gb300._lib import MoeError, MOE_ERR_RANGE
    with pytest.raises(MoeError) as ei:
        tiny.layer.test_withhold_ready(-2)
    assert ei.value.code == MOE_ERR_RANGE
    with pytest.raises(MoeError) as ei:
        tiny.layer.test_withhold_ready(1 << 20)
    assert ei.value.code == MOE_ERR_RANGE
