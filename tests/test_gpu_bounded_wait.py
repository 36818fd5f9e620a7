"""Failure detection on the device without a fault: every wait inside the
grouped GEMM is bounded, and a wait that runs out is reported in the call's
error word (PMOE_ERR_TIMEOUT) while the GPU context stays usable.

The test hook pmoe_debug_expire_gemm_wait makes the next grouped-GEMM launch
withhold one accumulator-full signal, so the epilogue waits on a barrier
that nothing completes; with a 2 ms limit the kernel gives up, records the
status and ends.  The next call, with the hook consumed, runs normally and
gives the same result as before."""
import numpy as np
import pytest
import torch

from precision_moe_adapter_gb300 import build, pmoe
from precision_moe_adapter_gb300 import inputs as gi
from precision_moe_adapter_gb300.layer import DeviceLayer
from helpers import t2np_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    pmoe.lib()


def dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if t.dtype == torch.uint16:
        t = t.view(torch.int16)
    return t.cuda()


def test_hook_rejects_unsafe_limits():
    for bad in (0, 10, 99_999, 3_000_000_000):
        with pytest.raises(pmoe.PmoeError):
            pmoe.pmoe_debug_expire_gemm_wait(bad)


def test_expired_wait_in_the_grouped_gemm():
    fmt, E, N, K = gi.INT4, 4, 256, 512
    q, s = gi.gen_matrix(fmt, E, N, K, seed=7, qsid="w2", ssid="s2")
    counts = np.array([300, 17, 0, 90])
    rows = int(counts.sum())
    A = gi.f32_to_bf16_bits(np.random.default_rng(7).standard_normal((rows, K)).astype(np.float32))
    offsets = dev(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32))
    qd, sd, Ad = dev(q), dev(s), dev(A)

    def run():
        out = torch.zeros((rows, N), dtype=torch.int16, device="cuda")
        ws = torch.zeros(pmoe.moe_grouped_gemm_ws_bytes(E, rows), dtype=torch.uint8, device="cuda")
        pmoe.moe_grouped_gemm(fmt, qd, sd, E, N, K, 0, Ad, offsets, rows, out, ws)
        return t2np_bits(out), pmoe.moe_query_status(ws)

    ref, st = run()
    assert st == pmoe.PMOE_OK
    pmoe.pmoe_debug_expire_gemm_wait(2_000_000)
    _, st = run()
    assert st == pmoe.PMOE_ERR_TIMEOUT
    again, st = run()                       # the hook was one-shot
    assert st == pmoe.PMOE_OK
    assert np.array_equal(again, ref)


def test_expired_wait_reported_by_the_layer():
    """Through the layer's forward: the status reaches moe_query_status of
    the forward's workspace, and the next forward matches the first."""
    cfg = gi.CONFIGS["tiny"]
    w13, s13, w2, s2 = gi.gen_weights(cfg)
    idx, w = gi.gen_routing(cfg)
    L = DeviceLayer(cfg, w13, s13, w2, s2)
    rt = L.new_routing()
    rt.idx.copy_(torch.from_numpy(idx))
    rt.w.copy_(torch.from_numpy(w))
    L.permute(rt)
    X = dev(gi.gen_x(cfg))
    Y0, Y1 = torch.empty_like(X), torch.empty_like(X)
    L.forward(X, rt, Y0)
    assert L.status() == pmoe.PMOE_OK
    pmoe.pmoe_debug_expire_gemm_wait(2_000_000)
    L.forward(X, rt, Y1)
    assert L.status() == pmoe.PMOE_ERR_TIMEOUT
    L.forward(X, rt, Y1)
    assert L.status() == pmoe.PMOE_OK
    assert torch.equal(Y0, Y1)
