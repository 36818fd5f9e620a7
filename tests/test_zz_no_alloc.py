"""moe_permute_noalloc: the grouping step without a caller workspace.

Its histogram lives in a fixed device buffer inside the library, shared by
every call, so the GPU test makes two calls in a row with different inputs
and checks each against moe_permute (bit-exact: the step is integer work).
The file sorts last so that it also runs after every other GPU test has
used the library in the same process.
"""
import ctypes

import numpy as np
import pytest
import torch

from precision_moe_adapter_gb300 import build, pmoe
from precision_moe_adapter_gb300 import inputs as gi

KEYS = ("counts", "offsets", "perm", "inv_perm", "active", "num_active")


def _bufs(T, E, k):
    i32 = dict(dtype=torch.int32, device="cuda")
    P = max(T * k, 1)
    b = dict(counts=torch.full((E,), 7, **i32), offsets=torch.full((E + 1,), 7, **i32),
             perm=torch.full((P,), 7, **i32), inv_perm=torch.full((P,), 7, **i32),
             active=torch.full((E,), 7, **i32), num_active=torch.full((1,), 7, **i32))
    rt = pmoe.routing(None, None, b["counts"], b["offsets"], b["perm"], b["inv_perm"],
                      b["active"], b["num_active"])
    return b, rt


def _host(b, P):
    out = {k_: v.cpu().numpy() for k_, v in b.items()}
    out["perm"], out["inv_perm"] = out["perm"][:P], out["inv_perm"][:P]
    return out


def test_oversized_problem_is_rejected_before_device_work():
    build.build()
    pmoe.lib()
    # ceil(65537 / 1024) * 4096 * 4 bytes > 1 MiB: refused on the host
    dm = pmoe.dims(65537, 64, 4096, 1, 64, 16)
    fake = 1 << 12   # never dereferenced: the size check comes first
    rt = pmoe.Routing(fake, fake, fake, fake, fake, fake, fake, fake)
    st = pmoe.lib().moe_permute_noalloc(dm, ctypes.c_void_p(fake), ctypes.byref(rt), None)
    assert st == pmoe.PMOE_ERR_WORKSPACE
    # just inside the limit: 64 blocks of 1024 pairs x 4096 experts = 1 MiB
    assert (65536 + 1023) // 1024 * 4096 * 4 == pmoe.PERMUTE_NOALLOC_SCRATCH_BYTES
    st = pmoe.lib().moe_permute_noalloc(pmoe.dims(8, 64, 8, 2, 64, 16), None, ctypes.byref(rt),
                                        None)
    assert st == pmoe.PMOE_ERR_INVALID_ARG   # T > 0 with no idx


@pytest.mark.gpu
def test_two_calls_in_a_row_match_moe_permute():
    build.build()
    pmoe.lib()
    # the last case fills the buffer exactly: 64 blocks of 1024 pairs x 4096
    # experts x 4 bytes = 1 MiB
    cases = [(8192, 384, 8, 1.1, 3), (777, 4096, 32, 1.1, 4), (2048, 4096, 32, 0.5, 5)]
    results = []
    for T, E, k, skew, seed in cases:
        cfg = gi.LayerConfig("p", T=T, d=64, E=E, k=k, I=64, b=16, seed=seed)
        idx, _ = gi.gen_routing(cfg, skew=skew)
        idx_d = torch.from_numpy(idx.astype(np.int32)).cuda()
        dm = pmoe.dims(T, 64, E, k, 64, 16)
        b, rt = _bufs(T, E, k)
        pmoe.moe_permute_noalloc(dm, idx_d, rt)
        torch.cuda.synchronize()
        results.append((dm, idx_d, _host(b, T * k), T, E, k))
    for dm, idx_d, got, T, E, k in results:
        b, rt = _bufs(T, E, k)
        ws = torch.zeros(max(pmoe.moe_workspace_bytes(dm, pmoe.OP_PERMUTE), 256),
                         dtype=torch.uint8, device="cuda")
        pmoe.moe_permute(dm, idx_d, rt, ws)
        assert pmoe.moe_query_status(ws) == pmoe.PMOE_OK
        want = _host(b, T * k)
        for key in KEYS:
            assert np.array_equal(got[key], want[key]), (T, E, key)
        assert int(got["offsets"][E]) == T * k


@pytest.mark.gpu
def test_bad_index_shows_in_the_outputs():
    build.build()
    pmoe.lib()
    idx = torch.tensor([[0, 1], [2, 9], [3, -1]], dtype=torch.int32, device="cuda")
    b, rt = _bufs(3, 8, 2)
    pmoe.moe_permute_noalloc(pmoe.dims(3, 64, 8, 2, 64, 16), idx, rt)
    got = _host(b, 6)
    assert got["counts"].sum() == 4 and got["offsets"][8] == 4
    assert got["inv_perm"][3] == -1 and got["inv_perm"][5] == -1
