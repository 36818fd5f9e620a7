"""Double-buffered adapter slots with an atomic switch: a forward reads the
slot control word once, so it uses one adapter version throughout even when
a publish lands on another stream while it runs."""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_adapter_gb300 import build, pmoe
from precision_moe_adapter_gb300 import inputs as gi
from precision_moe_adapter_gb300.layer import DeviceLayer

pytestmark = pytest.mark.gpu

CFG = gi.LayerConfig("slots", T=384, d=256, E=6, k=2, I=192, b=32, C=2, seed=21)


@pytest.fixture(scope="module")
def setup():
    build.build()
    pmoe.lib()
    cfg = CFG
    w13, s13, w2, s2 = gi.gen_weights(cfg)
    idx, w = gi.gen_routing(cfg)
    X = torch.from_numpy(gi.gen_x(cfg)).view(torch.int16).cuda()
    rb = lambda S: torch.from_numpy(gi.f32_to_bf16_bits(
        oracle.cayley(S.reshape(-1, cfg.b, cfg.b)).astype(np.float32)).reshape(S.shape)).view(torch.int16).cuda()
    ad = []
    for seed in (1, 2):
        Su = gi.gen_skew(cfg.E, cfg.d, cfg.b, seed, "S_up", 0.05)
        Sd = gi.gen_skew(cfg.E, cfg.I, cfg.b, seed, "S_down", 0.05)
        ad.append((rb(Su), rb(Sd)))
    host = dict(w13=w13, s13=s13, w2=w2, s2=s2, idx=idx, w=w, X=gi.gen_x(cfg),
                R=[tuple(t.cpu().numpy().view(np.uint16) for t in pair) for pair in ad])
    L = DeviceLayer(cfg, w13, s13, w2, s2)
    rt = L.new_routing()
    rt.idx.copy_(torch.from_numpy(idx))
    rt.w.copy_(torch.from_numpy(w))
    L.permute(rt)
    refs = []
    for Ru, Rd in ad:
        adp = pmoe.adapter(Ru, Rd, Ru[0].numel(), Rd[0].numel())
        Y = torch.empty_like(X)
        ws = L.workspace(pmoe.OP_FORWARD, cfg.C)
        pmoe.moe_chunked_forward(L.dims, L.wts, adp, rt.c(), X, cfg.C, pmoe.MODE_FUSED, Y, None, ws)
        refs.append(Y)
    torch.cuda.synchronize()
    ctrl = torch.zeros(1, dtype=torch.int64, device="cuda")
    slots = pmoe.adapter_slots(ad[0][0], ad[1][0], ad[0][1], ad[1][1], ad[0][0][0].numel(),
                               ad[0][1][0].numel(), ctrl)
    # the slot struct holds raw device pointers: keep their tensors alive
    return cfg, L, rt, X, refs, ctrl, slots, ad, host


def fwd(setup, Y, ver, stream=None):
    cfg, L, rt, X, refs, ctrl, slots, _, _ = setup
    ws = L.workspace(pmoe.OP_FORWARD, cfg.C)
    pmoe.moe_chunked_forward_slots(L.dims, L.wts, slots, rt.c(), X, cfg.C, pmoe.MODE_FUSED, Y,
                                   None, ver, ws, stream)


def test_each_slot_against_the_oracle(setup):
    """Each slot's forward against the oracle's layer with that slot's
    rotations, under the stated tolerance."""
    from helpers import assert_close, bits_to_f64
    cfg, L, rt, X, refs, ctrl, slots, _, h = setup
    for version in (8, 9):
        slot = version % 2
        pmoe.moe_adapter_publish(ctrl, slot, version)
        Y = torch.empty_like(X)
        fwd(setup, Y, None)
        torch.cuda.synchronize()
        Ru, Rd = h["R"][slot]
        OL = oracle.Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b, cfg.fmt, h["w13"], h["s13"],
                          h["w2"], h["s2"], R_up=Ru, R_down=Rd)
        _, Y64 = OL.forward(h["X"], h["idx"], h["w"])
        assert_close(bits_to_f64(Y.cpu().numpy().view(np.uint16)), Y64, f"slot {slot} Y")


def test_each_slot_is_the_single_adapter_forward(setup):
    cfg, L, rt, X, refs, ctrl, slots, _, _ = setup
    for version in (4, 5, 6):
        slot = version % 2
        pmoe.moe_adapter_publish(ctrl, slot, version)
        Y = torch.empty_like(X)
        ver = torch.zeros(1, dtype=torch.int32, device="cuda")
        fwd(setup, Y, ver)
        torch.cuda.synchronize()
        assert int(ver.item()) == version
        assert torch.equal(Y, refs[slot])
    assert L.status() == pmoe.PMOE_OK


def test_publishes_during_forwards_never_mix_versions(setup):
    """Forwards on one stream, publishes (version v -> slot v % 2) on
    another; each forward's output is the reference of the version it
    reports.  The time from a publish to the first forward that starts
    after it and uses it is the switch latency."""
    cfg, L, rt, X, refs, ctrl, slots, _, _ = setup
    n = 48
    Ys = [torch.empty_like(X) for _ in range(n)]
    vers = torch.zeros(n, dtype=torch.int32, device="cuda")
    s_fwd, s_pub = torch.cuda.Stream(), torch.cuda.Stream()
    ev_start = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ev_pub = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    pmoe.moe_adapter_publish(ctrl, 0, 100)
    torch.cuda.synchronize()
    for i in range(n):
        with torch.cuda.stream(s_fwd):
            ev_start[i].record(s_fwd)
            fwd(setup, Ys[i], vers[i:i + 1], s_fwd)
        with torch.cuda.stream(s_pub):
            # let a few forwards go by between publishes
            torch.cuda._sleep(20000)
            pmoe.moe_adapter_publish(ctrl, (101 + i) % 2, 101 + i, s_pub)
            ev_pub[i].record(s_pub)
    torch.cuda.synchronize()
    v = vers.cpu().numpy()
    for i in range(n):
        assert torch.equal(Ys[i], refs[int(v[i]) % 2]), (i, int(v[i]))
    assert np.all(np.diff(v) >= 0)               # versions only move forward
    lat = []
    for j in range(n):
        ver = 101 + j
        after = [i for i in range(n) if v[i] >= ver and ev_pub[j].elapsed_time(ev_start[i]) >= 0]
        if after:
            lat.append(min(ev_pub[j].elapsed_time(ev_start[i]) for i in after))
    print(f"versions seen: {len(set(v.tolist()))}; switch latency (ms): median "
          f"{np.median(lat) if lat else float('nan'):.3f}, max {max(lat) if lat else float('nan'):.3f}")
    assert len(set(v.tolist())) > 1
    assert L.status() == pmoe.PMOE_OK
