"""The allocation-free routing entry point (moe_route_static), called through
the C ABI, against the CPU oracle's router and against the routing of the
regular step (moe_decode_step) on the same rows.

moe_route_static exists for callers that may not allocate device memory when
they route: an engine whose GPU memory is all handed out by its own pool (or
planned before it starts) cannot have a library call cudaMalloc behind its
back, code running while a CUDA graph is being captured cannot call
cudaMalloc at all, and a caller that only wants routing decisions for rows it
already normalised should not need a full layer handle, which allocates the
whole step's scratch. Its scratch is a fixed array inside the library.

Calls in a row with different row counts must each give the oracle's top-k
ids exactly (inputs drawn with every top-k gap > 1e-3) and its weights within
1e-5 relative, and match the step's own routing; the later calls also show
that what an earlier call left in the shared array does not leak into the
next result. The full-size case (256 experts over 5120 columns, 48 rows) is
the shape closest to the array's size limit.

This file is collected last so that a run that stops at the first failure has
run every other test before it.
"""

import ctypes

import numpy as np
import pytest
import torch

from mxfp8_moe_decode_gb300 import _lib
from mxfp8_moe_decode_gb300 import workloads as W
from oracle import moe as O

from _harness import Layer, f64, gapped_tokens

pytestmark = pytest.mark.gpu

W_RTOL = 1e-5


def _route(normed, gate_w, bias, k, dev):
    """One moe_route_static call on the current stream; returns (ids, weights)
    on the host after the stream has finished."""
    m, hidden = normed.shape
    experts = gate_w.shape[0]
    ids = torch.full((m, k), -1, dtype=torch.int32, device=dev)
    wts = torch.full((m, k), -1.0, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    rc = _lib.lib().moe_route_static(normed.data_ptr(), gate_w.data_ptr(), bias.data_ptr(), m,
                                     hidden, experts, k, ids.data_ptr(), wts.data_ptr(),
                                     ctypes.c_void_p(stream.cuda_stream))
    assert rc == _lib.MOE_OK, rc
    st = _lib.lib().moe_route_static_status(ctypes.c_void_p(stream.cuda_stream))
    assert st == _lib.MOE_OK, st
    return ids.cpu().numpy(), wts.cpu().numpy()


def test_route_static_matches_oracle_and_step_routing():
    L = Layer(W.WORKLOADS["tiny_m1"])
    try:
        d = L.wl.dims
        dev = L.dev
        gate_w = L.ri["gate_w"].to(dev)
        bias = L.ri["bias"].to(dev)
        for m in (1, 4, 48, 5):  # calls in a row, different sizes
            x, _ = gapped_tokens(L.wl, L.ri, m=m)
            dbg = L.layer.debug_buffers(m)
            L.layer.step(x.to(dev), debug=dbg)
            ids, wts = _route(dbg["normed"], gate_w, bias, d.topk, dev)
            rt = O.router(f64(dbg["normed"]), f64(L.ri["gate_w"]), f64(L.ri["bias"]), d.topk)
            assert np.array_equal(ids, rt.ids), m
            np.testing.assert_allclose(wts, rt.weights, rtol=W_RTOL)
            assert np.array_equal(ids, dbg["topk_ids"].cpu().numpy()), m
            np.testing.assert_allclose(wts, dbg["topk_w"].cpu().numpy(), rtol=W_RTOL)
        assert L.layer.status() == 0
    finally:
        L.close()


def test_route_static_full_size_router():
    # the full-size router (256 experts, 5120 columns, top-8) on 48 gapped
    # rows, then on a 16-row prefix: no layer handle at all
    wl = W.WORKLOADS["full_m48_uniform"]
    d = wl.dims
    dev = torch.device("cuda:0")
    ri = W.router_inputs(wl)
    x, _ = gapped_tokens(wl, ri)
    normed64 = O.rmsnorm(f64(x), f64(ri["norm_w"]), d.eps)  # bf16 values
    normed = torch.from_numpy(normed64).to(torch.bfloat16).to(dev)
    gate_w = ri["gate_w"].to(dev)
    bias = ri["bias"].to(dev)
    rt = O.router(normed64, f64(ri["gate_w"]), f64(ri["bias"]), d.topk)
    for m in (48, 16):
        ids, wts = _route(normed[:m].contiguous(), gate_w, bias, d.topk, dev)
        assert np.array_equal(ids, rt.ids[:m]), m
        np.testing.assert_allclose(wts, rt.weights[:m], rtol=W_RTOL)


def test_route_static_in_a_cuda_graph():
    # The call's scratch is the library's fixed array, so it can be captured:
    # captured once and replayed, it gives the uncaptured call's ids and
    # weights bit for bit; its status call refuses while the stream captures
    # (it would have to synchronise), and so does a layer's.
    wl = W.WORKLOADS["full_m16"]
    d = wl.dims
    dev = torch.device("cuda:0")
    ri = W.router_inputs(wl)
    x, _ = gapped_tokens(wl, ri)
    normed64 = O.rmsnorm(f64(x), f64(ri["norm_w"]), d.eps)
    normed = torch.from_numpy(normed64).to(torch.bfloat16).to(dev)
    gate_w = ri["gate_w"].to(dev)
    bias = ri["bias"].to(dev)
    m = normed.shape[0]
    ids0, wts0 = _route(normed, gate_w, bias, d.topk, dev)  # outside capture first

    ids = torch.full((m, d.topk), -1, dtype=torch.int32, device=dev)
    wts = torch.full((m, d.topk), -1.0, dtype=torch.float32, device=dev)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    L = Layer(W.WORKLOADS["tiny_m1"])
    try:
        xt = gapped_tokens(L.wl, L.ri, m=2)[0].to(dev)
        with torch.cuda.stream(s):
            L.layer.step(xt, stream=s)  # the layer's last stream is s
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                rc = _lib.lib().moe_route_static(normed.data_ptr(), gate_w.data_ptr(), bias.data_ptr(),
                                                 m, d.hidden, d.experts, d.topk, ids.data_ptr(),
                                                 wts.data_ptr(), ctypes.c_void_p(s.cuda_stream))
                st = _lib.lib().moe_route_static_status(ctypes.c_void_p(s.cuda_stream))
                layer_st = L.layer.status()
        assert rc == _lib.MOE_OK, rc
        assert st == _lib.MOE_ERR_CAPTURE, st
        assert layer_st == _lib.MOE_ERR_CAPTURE, layer_st
        assert torch.all(ids == -1)  # nothing ran during capture
        g.replay()
        torch.cuda.synchronize(dev)
        assert np.array_equal(ids.cpu().numpy(), ids0)
        assert np.array_equal(wts.cpu().numpy(), wts0)  # bit for bit
        assert _lib.lib().moe_route_static_status(ctypes.c_void_p(s.cuda_stream)) == _lib.MOE_OK
        assert L.layer.status() == _lib.MOE_OK
    finally:
        L.close()


def test_route_static_refuses_oversized_and_bad_args():
    fn = _lib.lib().moe_route_static
    p = 0x10000  # never dereferenced: every call below is refused on the host
    # experts 512 with hidden 8192 needs more scratch than the fixed array holds
    assert fn(p, p, p, 48, 8192, 512, 8, p, p, None) == _lib.MOE_ERR_UNSUPPORTED
    assert fn(p, p, p, 0, 1024, 64, 4, p, p, None) == _lib.MOE_ERR_RANGE
    assert fn(p, p, p, 49, 1024, 64, 4, p, p, None) == _lib.MOE_ERR_RANGE
    assert fn(None, p, p, 4, 1024, 64, 4, p, p, None) == _lib.MOE_ERR_ARG
    assert fn(p + 8, p, p, 4, 1024, 64, 4, p, p, None) == _lib.MOE_ERR_ALIGN
