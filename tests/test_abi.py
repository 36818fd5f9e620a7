"""The C ABI on the host: the library builds, loads without a GPU, exports
every function that include/pmoe.h declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

from precision_moe_adapter_gb300 import build, pmoe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return pmoe.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "pmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert set(pmoe.EXPORTS) <= set(names)


def test_status_strings(L):
    for s in range(7):
        assert pmoe.status_string(s)


def _d(**kw):
    base = dict(T=64, d=256, E=8, k=2, inter=128, block=32)
    base.update(kw)
    return pmoe.Dims(*[base[f] for f in ("T", "d", "E", "k", "inter", "block")])


def test_workspace_sizes(L):
    d = _d()
    for op in (pmoe.OP_PERMUTE, pmoe.OP_FORWARD, pmoe.OP_BACKWARD):
        assert pmoe.moe_workspace_bytes(d, op, 4, pmoe.MODE_FUSED) > 256
    f = pmoe.moe_workspace_bytes(d, pmoe.OP_FORWARD, 4, pmoe.MODE_FUSED)
    s = pmoe.moe_workspace_bytes(d, pmoe.OP_FORWARD, 4, pmoe.MODE_SCRATCH)
    assert s - f >= pmoe.moe_scratch_bytes(d, 4, pmoe.MODE_SCRATCH)
    assert pmoe.moe_scratch_bytes(d, 4, pmoe.MODE_SCRATCH) == 4 * 3 * 128 * 256 * 2
    assert pmoe.moe_scratch_bytes(d, 4, pmoe.MODE_FUSED) == 0
    assert pmoe.moe_scratch_bytes(d, 100, pmoe.MODE_SCRATCH) == 8 * 3 * 128 * 256 * 2
    assert pmoe.moe_workspace_bytes(_d(d=100), pmoe.OP_FORWARD, 4, 0) == 0


@pytest.mark.parametrize("bad", [dict(d=100), dict(inter=96), dict(block=24), dict(k=9),
                                 dict(E=5000), dict(k=0), dict(T=-1), dict(block=128, d=192)])
def test_invalid_dims_rejected(L, bad):
    d = _d(**bad)
    st = L.moe_route(d, None, None, None, None, None, None, 0, None, 0, None)
    assert st == pmoe.PMOE_ERR_INVALID_ARG


def test_validation_before_device(L):
    d = _d()
    # missing workspace
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    assert L.moe_route(d, p, p, None, None, p, p, 0, None, 0, None) == pmoe.PMOE_ERR_WORKSPACE
    # misaligned pointer
    assert L.moe_route(d, p + 2, p, None, None, p, p, 0, p, 1 << 30, None) == pmoe.PMOE_ERR_INVALID_ARG
    # bad weight format / chunk size / mode
    w = pmoe.Weights(7, p, p, p, p)
    rt = pmoe.Routing(p, p, p, p, p, p, p, p)
    assert L.moe_chunked_forward(d, ctypes.byref(w), None, ctypes.byref(rt), p, 4, 0, p, None, p,
                                 1 << 30, None) == pmoe.PMOE_ERR_INVALID_ARG
    w = pmoe.Weights(0, p, p, p, p)
    assert L.moe_chunked_forward(d, ctypes.byref(w), None, ctypes.byref(rt), p, 0, 0, p, None, p,
                                 1 << 30, None) == pmoe.PMOE_ERR_INVALID_ARG
    assert L.moe_chunked_forward(d, ctypes.byref(w), None, ctypes.byref(rt), p, 4, 9, p, None, p,
                                 1 << 30, None) == pmoe.PMOE_ERR_INVALID_ARG
    # FP8 needs multiples of 128
    w8 = pmoe.Weights(2, p, p, p, p)
    assert L.moe_chunked_forward(_d(inter=192), ctypes.byref(w8), None, ctypes.byref(rt), p, 4, 0,
                                 p, None, p, 1 << 30, None) == pmoe.PMOE_ERR_INVALID_ARG
    # adapter: R_down without R_up
    a = pmoe.Adapter(None, p, 0, 0)
    assert L.moe_chunked_forward(d, ctypes.byref(w), ctypes.byref(a), ctypes.byref(rt), p, 4, 0, p,
                                 None, p, 1 << 30, None) == pmoe.PMOE_ERR_INVALID_ARG
    # backward: adapter gradient buffers required with an adapter
    a = pmoe.Adapter(p, p, 0, 0)
    assert L.moe_backward_data(d, ctypes.byref(w), ctypes.byref(a), ctypes.byref(rt), p, p, p, 4,
                               p, None, None, None, p, 1 << 30, None) == pmoe.PMOE_ERR_INVALID_ARG
    # dequant shape rules
    assert L.moe_dequant(0, p, p, 4, 48, p, None) == pmoe.PMOE_ERR_INVALID_ARG
    assert L.moe_dequant(2, p, p, 64, 128, p, None) == pmoe.PMOE_ERR_INVALID_ARG
    assert L.adapter_apply(4, 96, 64, p, p, p, None) == pmoe.PMOE_ERR_INVALID_ARG
    assert L.adapter_apply(4, 64, 16, p, p, p, None) == pmoe.PMOE_ERR_INVALID_ARG   # aliasing
    assert L.adapter_cayley(4, 256, p, p, None, None) == pmoe.PMOE_ERR_INVALID_ARG
    # empty inputs are valid no-ops
    assert L.moe_dequant(0, None, None, 0, 64, None, None) == pmoe.PMOE_OK
    assert L.adapter_cayley(0, 16, None, None, None, None) == pmoe.PMOE_OK
