"""The C-ABI library loads and exports every entry point include/moe_decode.h
declares; argument checks that need no GPU (CPU only)."""

import ctypes
import os
import re

import pytest

from mxfp8_moe_decode_gb300 import _lib
from mxfp8_moe_decode_gb300._lib import (MOE_ERR_ALIGN, MOE_ERR_ARG, MOE_ERR_RANGE,
                                         MOE_ERR_UNSUPPORTED, MOE_OK, MoeConfig, MoeWeights)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_decode.h")


@pytest.fixture(scope="module")
def L():
    from mxfp8_moe_decode_gb300 import build
    build.build()
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "moe_create" in names and "moe_decode_step" in names and "moe_destroy" in names
    for n in names:
        assert hasattr(L, n), n


def test_kernel_names(L):
    n = L.moe_kernel_count()
    assert n == 5
    names = [L.moe_kernel_name(i).decode() for i in range(n)]
    assert names == ["seam", "router", "topk", "experts", "combine"]
    assert L.moe_kernel_name(n) is None


def test_strerror(L):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert L.moe_strerror(code)
    assert L.moe_strerror(MOE_OK) == b"ok"


def _cfg(**kw):
    c = dict(hidden=1024, experts=64, topk=4, inter=512, shared_inter=512, max_tokens=48,
             eps=1e-6)
    c.update(kw)
    return MoeConfig(**c)


def _weights(base=0x10000):
    return MoeWeights(*[base + 0x1000 * i for i in range(11)])


def test_create_rejects_bad_config_without_touching_a_gpu(L):
    h = ctypes.c_void_p()
    w = _weights()
    assert L.moe_create(None, ctypes.byref(w), 0, ctypes.byref(h)) == MOE_ERR_ARG
    bad = [dict(hidden=1000), dict(hidden=128), dict(experts=48), dict(topk=17),
           dict(topk=0), dict(inter=500), dict(shared_inter=1024), dict(max_tokens=49),
           dict(experts=1024)]
    for kw in bad:
        rc = L.moe_create(ctypes.byref(_cfg(**kw)), ctypes.byref(w), 0, ctypes.byref(h))
        assert rc in (MOE_ERR_UNSUPPORTED, MOE_ERR_ARG), (kw, rc)
        assert h.value is None
    wn = _weights()
    wn.w13 = None
    assert L.moe_create(ctypes.byref(_cfg()), ctypes.byref(wn), 0, ctypes.byref(h)) == MOE_ERR_ARG
    wa = _weights()
    wa.w2 = 0x10008
    assert L.moe_create(ctypes.byref(_cfg()), ctypes.byref(wa), 0, ctypes.byref(h)) == MOE_ERR_ALIGN


def test_step_rejects_null_handle_and_range(L):
    assert L.moe_decode_step(None, 0x1000, 1, 0x2000, None, None) == MOE_ERR_ARG
    assert L.moe_status(None) == MOE_ERR_ARG
    assert L.moe_clear_status(None) == MOE_ERR_ARG
    v = ctypes.c_int()
    assert L.moe_last_unique_experts(None, ctypes.byref(v)) == MOE_ERR_ARG
    assert L.moe_scratch_bytes(None) == 0
    L.moe_destroy(None)
    assert MOE_ERR_RANGE == -2


def test_attn_seam_argument_checks_without_a_gpu(L):
    f = L.moe_attn_seam_x8
    x, w, b, c, y = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    assert f(None, w, 4, 256, 1e-6, b, c, y, None) == MOE_ERR_ARG
    assert f(x, w, 4, 256, 1e-6, b, None, y, None) == MOE_ERR_ARG
    assert f(x + 8, w, 4, 256, 1e-6, b, c, y, None) == MOE_ERR_ALIGN
    assert f(x, w, 4, 256, 1e-6, b + 4, c, y, None) == MOE_ERR_ALIGN
    assert f(x, w, 4, 256, 1e-6, b, c, y + 4, None) == MOE_ERR_ALIGN
    assert f(x, w, 0, 256, 1e-6, b, c, y, None) == MOE_ERR_RANGE
    assert f(x, w, 49, 256, 1e-6, b, c, y, None) == MOE_ERR_RANGE
    for h in (0, 16, 1000, 8224):
        assert f(x, w, 4, h, 1e-6, b, c, y, None) == MOE_ERR_UNSUPPORTED, h
    assert f(x, w, 4, 256, -1.0, b, c, y, None) == MOE_ERR_ARG
    assert f(x, w, 4, 256, float("nan"), b, c, y, None) == MOE_ERR_ARG


def test_create_checks_the_routed_format_without_a_gpu(L):
    h = ctypes.c_void_p()
    w = _weights()
    rc = L.moe_create(ctypes.byref(_cfg(routed_format=2)), ctypes.byref(w), 0, ctypes.byref(h))
    assert rc == MOE_ERR_UNSUPPORTED and h.value is None
    # MXFP4 routed weights must start on 32 bytes (the 4-bit tensor copies)
    for key in ("w13", "w2"):
        wa = _weights()
        setattr(wa, key, 0x10010)
        rc = L.moe_create(ctypes.byref(_cfg(routed_format=1)), ctypes.byref(wa), 0, ctypes.byref(h))
        assert rc == MOE_ERR_ALIGN and h.value is None, key


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """The binding only loads the in-tree library: without it every entry
    raises instead of falling back to anything else."""
    import mxfp8_moe_decode_gb300.api as api
    monkeypatch.setattr(_lib, "_LIB", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent" / "libmoe_decode.so"))
    with pytest.raises(FileNotFoundError):
        _lib.lib()
    with pytest.raises(FileNotFoundError):
        api.kernel_names()
