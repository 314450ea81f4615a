"""The allocation-free routing entry point (moe_route_static), called through
the C ABI, against the routing of the regular step (moe_decode_step) on the
same rows.

moe_route_static exists for callers that may not allocate device memory when
they route (a memory pool that owns the whole GPU, a CUDA graph capture in
progress, a caller without a full layer handle): its scratch is a fixed array
inside the library. Two calls in a row with different row counts must each
match the step's own top-k ids exactly and its weights within the tolerance
the parity tests use (1e-5 relative); the second call also shows that what
the first call left in the shared array does not leak into the next result.

This file is collected last so that a run that stops at the first failure has
run every other test before it.
"""

import ctypes

import numpy as np
import pytest
import torch

from mxfp8_moe_decode_gb300 import _lib
from mxfp8_moe_decode_gb300 import workloads as W

from _harness import Layer, gapped_tokens

pytestmark = pytest.mark.gpu

W_RTOL = 1e-5


def _route_static():
    fn = _lib.lib().moe_route_static
    vp, ip = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, ip, ip, ip, ip, vp, vp, vp]
    fn.restype = ip
    return fn


def test_route_static_matches_step_routing():
    fn = _route_static()
    L = Layer(W.WORKLOADS["tiny_m1"])
    try:
        d = L.wl.dims
        dev = L.dev
        gate_w = L.ri["gate_w"].to(dev)
        bias = L.ri["bias"].to(dev)
        stream = torch.cuda.current_stream(dev)
        for m in (5, 48):  # two calls in a row, different sizes
            x, _ = gapped_tokens(L.wl, L.ri, m=m)
            dbg = L.layer.debug_buffers(m)
            L.layer.step(x.to(dev), debug=dbg)
            ids = torch.full((m, d.topk), -1, dtype=torch.int32, device=dev)
            wts = torch.full((m, d.topk), -1.0, dtype=torch.float32, device=dev)
            rc = fn(dbg["normed"].data_ptr(), gate_w.data_ptr(), bias.data_ptr(), m, d.hidden,
                    d.experts, d.topk, ids.data_ptr(), wts.data_ptr(),
                    ctypes.c_void_p(stream.cuda_stream))
            assert rc == _lib.MOE_OK, rc
            torch.cuda.synchronize(dev)
            assert np.array_equal(ids.cpu().numpy(), dbg["topk_ids"].cpu().numpy()), m
            np.testing.assert_allclose(wts.cpu().numpy(), dbg["topk_w"].cpu().numpy(),
                                       rtol=W_RTOL)
        assert L.layer.status() == 0
    finally:
        L.close()


def test_route_static_refuses_oversized_and_bad_args():
    fn = _route_static()
    p = 0x10000  # never dereferenced: every call below is refused on the host
    # experts 512 with hidden 8192 needs more scratch than the fixed array holds
    assert fn(p, p, p, 48, 8192, 512, 8, p, p, None) == _lib.MOE_ERR_UNSUPPORTED
    assert fn(p, p, p, 0, 1024, 64, 4, p, p, None) == _lib.MOE_ERR_RANGE
    assert fn(p, p, p, 49, 1024, 64, 4, p, p, None) == _lib.MOE_ERR_RANGE
    assert fn(None, p, p, 4, 1024, 64, 4, p, p, None) == _lib.MOE_ERR_ARG
    assert fn(p + 8, p, p, 4, 1024, 64, 4, p, p, None) == _lib.MOE_ERR_ALIGN
