"""SCRATCH mode: the pages' literal scheme (dequantize the C experts of a
chunk into a global BF16 buffer, run the chunk's grouped GEMMs, reuse the
buffer for the next chunk).  Its peak dequant scratch is C x 3 x inter x d
BF16 (the gate, up and down matrices of C experts), and it lives in the
caller's workspace: moe_scratch_bytes reports it, the workspace grows by
exactly that much over FUSED mode, the device memory the workspace takes
matches, and the forward call itself takes no device memory."""
import numpy as np
import pytest
import torch

from precision_moe_adapter_gb300 import build, pmoe
from precision_moe_adapter_gb300 import inputs as gi
from precision_moe_adapter_gb300.layer import DeviceLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    pmoe.lib()


def free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


@pytest.mark.parametrize("C", [1, 8, 32, 384])
def test_scratch_bytes_in_the_workspace_and_device_memory(C):
    cfg = gi.CONFIGS["kimi_k2"].with_(T=64)
    dm = pmoe.dims(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b)
    want = min(C, cfg.E) * 3 * cfg.I * cfg.d * 2
    assert pmoe.moe_scratch_bytes(dm, C, pmoe.MODE_SCRATCH) == want
    assert pmoe.moe_scratch_bytes(dm, C, pmoe.MODE_FUSED) == 0
    fused = pmoe.moe_workspace_bytes(dm, pmoe.OP_FORWARD, C, pmoe.MODE_FUSED)
    scr = pmoe.moe_workspace_bytes(dm, pmoe.OP_FORWARD, C, pmoe.MODE_SCRATCH)
    assert 0 <= scr - fused - want < 256          # one 256-byte aligned region
    torch.cuda.empty_cache()
    f0 = free_bytes()
    ws = torch.empty(scr, dtype=torch.uint8, device="cuda")
    taken = f0 - free_bytes()
    # the allocator rounds a large block up to whole 2 MiB pages
    assert scr <= taken <= scr + (32 << 20), (scr, taken)
    del ws
    torch.cuda.empty_cache()


def test_forward_takes_no_device_memory():
    """A SCRATCH-mode forward (and a FUSED one) with its workspace in place
    changes the free device memory by nothing: the library allocates none."""
    cfg = gi.CONFIGS["tiny"]
    w13, s13, w2, s2 = gi.gen_weights(cfg)
    idx, w = gi.gen_routing(cfg)
    L = DeviceLayer(cfg, w13, s13, w2, s2)
    rt = L.new_routing()
    rt.idx.copy_(torch.from_numpy(idx))
    rt.w.copy_(torch.from_numpy(w))
    L.permute(rt)
    X = torch.from_numpy(gi.gen_x(cfg)).view(torch.int16).cuda()
    Y0, Y1 = torch.empty_like(X), torch.empty_like(X)
    for mode in (pmoe.MODE_SCRATCH, pmoe.MODE_FUSED):
        L.workspace(pmoe.OP_FORWARD, cfg.C, mode)      # allocated beforehand
    L.forward(X, rt, Y0, mode=pmoe.MODE_SCRATCH)      # first call: lazy module setup
    L.forward(X, rt, Y1, mode=pmoe.MODE_FUSED)
    f0 = free_bytes()
    L.forward(X, rt, Y0, mode=pmoe.MODE_SCRATCH)
    L.forward(X, rt, Y1, mode=pmoe.MODE_FUSED)
    assert free_bytes() == f0
    assert torch.equal(Y0, Y1)
    assert L.status() == pmoe.PMOE_OK
