"""GPU parity of the whole layer against the oracle: forward Y and the
backward-data outputs (dX, d_topk_w, dR_up, dR_down) within the stated
tolerance, on sizes that span several tiles with ragged tails; and the
invariants the pages fix: chunk size and mode do not change the result,
a zero adapter is the frozen base (the reference policy), the base takes
no update, and the reductions are deterministic."""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_adapter_gb300 import build, pmoe
from precision_moe_adapter_gb300 import inputs as gi
from precision_moe_adapter_gb300.layer import DeviceLayer
from helpers import assert_close, bits_to_f64, check_cayley, t2np_bits

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


def rbits(S):
    """BF16 rotation blocks from the oracle's Cayley map of S."""
    b = S.shape[-1]
    return gi.f32_to_bf16_bits(oracle.cayley(S.reshape(-1, b, b)).astype(np.float32)).reshape(S.shape)


def make_case(cfg, skew=1.1):
    c = dict(cfg=cfg, X=gi.gen_x(cfg), dY=gi.gen_dy(cfg))
    c["w13"], c["s13"], c["w2"], c["s2"] = gi.gen_weights(cfg)
    c["idx"], c["w"] = gi.gen_routing(cfg, skew=skew)
    Su, Sd = gi.gen_adapter_params(cfg)
    c["R_up"] = None if Su is None else rbits(Su)
    c["R_down"] = None if Sd is None else rbits(Sd)
    return c


def run_gpu(c, C=None, mode=pmoe.MODE_FUSED, backward=True, R_up="case", R_down="case"):
    cfg = c["cfg"]
    R_up = c["R_up"] if isinstance(R_up, str) else R_up
    R_down = c["R_down"] if isinstance(R_down, str) else R_down
    L = DeviceLayer(cfg, c["w13"], c["s13"], c["w2"], c["s2"], R_up=R_up, R_down=R_down)
    rt = L.new_routing()
    rt.idx.copy_(torch.from_numpy(c["idx"]))
    rt.w.copy_(torch.from_numpy(c["w"]))
    L.permute(rt)
    X = dev(c["X"])
    Y = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device="cuda")
    ctx = L.new_ctx()
    L.forward(X, rt, Y, C=C, mode=mode, ctx=ctx)
    out = dict(Y=t2np_bits(Y))
    # the saved h and h~ rows (expert-sorted) and each row's expert
    P, I = cfg.P, cfg.I
    hb = ctx[P * 2 * I * 4:P * 2 * I * 4 + 2 * P * I * 2].view(torch.int16).view(2, P, I)
    hb = hb.cpu().numpy().view(np.uint16)
    out["h"], out["ht"] = hb[0], hb[1]
    out["offsets"] = rt.offsets.cpu().numpy()
    if backward:
        dX = torch.empty_like(Y)
        dtw = torch.zeros((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
        dRu, dRd = L.grads()
        L.backward(X, dev(c["dY"]), ctx, rt, dX, dtw, dRu, dRd, C=C)
        out.update(dX=t2np_bits(dX), dtw=dtw.cpu().numpy(),
                   dR_up=None if dRu is None else dRu.cpu().numpy(),
                   dR_down=None if dRd is None else dRd.cpu().numpy())
    torch.cuda.synchronize()
    assert L.status() == pmoe.PMOE_OK
    out["layer"] = L
    return out


def run_oracle(c, backward=True):
    cfg = c["cfg"]
    L = oracle.Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b, cfg.fmt, c["w13"], c["s13"],
                     c["w2"], c["s2"], R_up=c["R_up"], R_down=c["R_down"])
    Y, Y64 = L.forward(c["X"], c["idx"], c["w"])
    out = dict(Y=Y, Y64=Y64)
    if backward:
        out.update(L.backward(c["X"], c["dY"], c["idx"], c["w"]))
    return out


CASES = {
    "int4_medium": gi.LayerConfig("m", T=384, d=256, E=6, k=2, I=192, b=32, C=2),
    "int4_b64_k3": gi.LayerConfig("m", T=200, d=384, E=5, k=3, I=256, b=64, C=2, seed=1),
    "mxfp4": gi.LayerConfig("m", T=160, d=256, E=4, k=2, I=128, b=32, fmt=gi.MXFP4, C=3, seed=2),
    "fp8": gi.LayerConfig("m", T=96, d=256, E=4, k=2, I=256, b=64, fmt=gi.FP8, C=2, seed=3),
    "shared_adapter": gi.LayerConfig("m", T=130, d=256, E=5, k=2, I=128, b=16, C=2,
                                     adapter="shared", seed=4),
    "no_adapter": gi.LayerConfig("m", T=100, d=192, E=4, k=2, I=128, b=32, C=4,
                                 adapter="none", seed=5),
    "ragged_T37": gi.LayerConfig("m", T=37, d=128, E=7, k=3, I=64, b=32, C=3, seed=6),
    "decode_T1": gi.LayerConfig("m", T=1, d=256, E=16, k=4, I=128, b=64, C=8, seed=7),
    "dense_E1": gi.LayerConfig("m", T=70, d=128, E=1, k=1, I=128, b=128, C=1, seed=8),
    "tiny": gi.CONFIGS["tiny"],
}


@pytest.mark.parametrize("name", list(CASES))
def test_forward_backward_parity(name):
    c = make_case(CASES[name])
    g = run_gpu(c)
    o = run_oracle(c)
    assert_close(bits_to_f64(g["Y"]), o["Y64"], f"{name} Y")
    if c["R_down"] is not None and CASES[name].b <= 64:
        # h~ = bf16(h R_down[e]) rounded as the exact sum is, per expert
        # (b <= 64: the rotations' exact rounding)
        off, b = g["offsets"], CASES[name].b
        for e in range(CASES[name].E):
            r0, r1 = off[e], off[e + 1]
            if r1 > r0:
                Re = c["R_down"][0 if CASES[name].adapter == "shared" else e]
                assert np.array_equal(g["ht"][r0:r1], oracle.adapter_apply(g["h"][r0:r1], Re, b)), e
    assert_close(bits_to_f64(g["dX"]), o["dX64"], f"{name} dX")
    assert_close(g["dtw"], o["d_topk_w"], f"{name} d_topk_w")
    if c["R_up"] is not None:
        assert_close(g["dR_up"], o["dR_up"], f"{name} dR_up")
        assert_close(g["dR_down"], o["dR_down"], f"{name} dR_down")


def test_chunk_size_and_mode_do_not_change_results():
    c = make_case(CASES["int4_medium"])
    ref = run_gpu(c, C=1)
    for C, mode in ((2, pmoe.MODE_FUSED), (6, pmoe.MODE_FUSED), (100, pmoe.MODE_FUSED),
                    (1, pmoe.MODE_SCRATCH), (4, pmoe.MODE_SCRATCH), (6, pmoe.MODE_SCRATCH)):
        g = run_gpu(c, C=C, mode=mode)
        for key in ("Y", "dX", "dtw", "dR_up", "dR_down"):
            assert np.array_equal(g[key], ref[key]), (C, mode, key)


def test_zero_adapter_is_the_frozen_base():
    """S = 0 (R = I from the device Cayley map) reproduces the adapter-less
    layer bit for bit: the reference policy of the pages."""
    cfg = CASES["int4_medium"]
    c = make_case(cfg)
    b = cfg.b
    S0 = torch.zeros((cfg.E, cfg.d // b, b, b), dtype=torch.float32, device="cuda")
    Ru = torch.empty(S0.shape, dtype=torch.int16, device="cuda")
    pmoe.adapter_cayley(S0.numel() // (b * b), b, S0, Ru, None)
    S1 = torch.zeros((cfg.E, cfg.I // b, b, b), dtype=torch.float32, device="cuda")
    Rd = torch.empty(S1.shape, dtype=torch.int16, device="cuda")
    pmoe.adapter_cayley(S1.numel() // (b * b), b, S1, Rd, None)
    torch.cuda.synchronize()
    eye = gi.f32_to_bf16_bits(np.eye(b, dtype=np.float32))
    assert np.all(t2np_bits(Ru) == eye) and np.all(t2np_bits(Rd) == eye)
    on = run_gpu(c, R_up=t2np_bits(Ru), R_down=t2np_bits(Rd))
    off = run_gpu(c, R_up=None, R_down=None)
    assert np.array_equal(on["Y"], off["Y"])
    assert np.array_equal(on["dX"], off["dX"])
    assert np.array_equal(on["dtw"], off["dtw"])


def test_runs_are_deterministic_and_base_is_untouched():
    c = make_case(CASES["int4_b64_k3"])
    a = run_gpu(c)
    L = a["layer"]
    before = [t.clone() for t in (L.w13, L.s13, L.w2, L.s2)]
    b = run_gpu(c)
    for key in ("Y", "dX", "dtw", "dR_up", "dR_down"):
        assert np.array_equal(a[key], b[key]), key
    # the frozen base is read-only for the layer: no base weight gradient,
    # no write into the weight buffers
    X = dev(c["X"])
    rt = L.new_routing()
    rt.idx.copy_(torch.from_numpy(c["idx"]))
    rt.w.copy_(torch.from_numpy(c["w"]))
    L.permute(rt)
    Y = torch.empty((c["cfg"].T, c["cfg"].d), dtype=torch.int16, device="cuda")
    ctx = L.new_ctx()
    L.forward(X, rt, Y, ctx=ctx)
    dX = torch.empty_like(Y)
    L.backward(X, dev(c["dY"]), ctx, rt, dX, None, *L.grads())
    torch.cuda.synchronize()
    for t0, t1 in zip(before, (L.w13, L.s13, L.w2, L.s2)):
        assert torch.equal(t0, t1)


def test_tiny_end_to_end_from_the_router():
    """The tiny configuration from X: device router (exact mode) -> grouping
    -> forward -> backward, against the oracle with its canonical-order
    routing, which the device reproduces bit for bit."""
    cfg = gi.CONFIGS["tiny"]
    X, dY = gi.gen_x(cfg), gi.gen_dy(cfg)
    w13, s13, w2, s2 = gi.gen_weights(cfg)
    Wr, bias = gi.gen_router(cfg)
    Su, Sd = gi.gen_adapter_params(cfg)
    # the device Cayley map of S, checked on its own; the layer then takes
    # the oracle's BF16 rotations, so both sides multiply by the same R
    Ld = DeviceLayer(cfg, w13, s13, w2, s2, S_up=Su, S_down=Sd)
    torch.cuda.synchronize()
    for S, Rb_, Rf_ in ((Su, Ld.R_up, Ld.Rf_up), (Sd, Ld.R_down, Ld.Rf_down)):
        check_cayley(t2np_bits(Rb_).reshape(-1, cfg.b, cfg.b), Rf_.cpu().numpy().reshape(-1, cfg.b, cfg.b),
                     oracle.cayley(S.reshape(-1, cfg.b, cfg.b)), cfg.b)
    Ru, Rd = rbits(Su), rbits(Sd)
    L = DeviceLayer(cfg, w13, s13, w2, s2, Wr=Wr, bias=bias, R_up=Ru, R_down=Rd)
    rt = L.new_routing()
    Xd = dev(X)
    logits = torch.zeros((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    L.route(Xd, rt, logits, mode=pmoe.ROUTE_EXACT)
    L.permute(rt)
    Y = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device="cuda")
    ctx = L.new_ctx()
    L.forward(Xd, rt, Y, ctx=ctx)
    dX = torch.empty_like(Y)
    L.backward(Xd, dev(dY), ctx, rt, dX, None, *L.grads())
    torch.cuda.synchronize()
    assert L.status() == pmoe.PMOE_OK
    # the exact router mode: logits, selection and weights equal the oracle's
    # canonical-order routing for every token
    o_logits = oracle.route_canonical(X, Wr, bias)
    o_idx, o_w = oracle.topk(o_logits, cfg.k)
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), o_logits.view(np.uint32))
    assert np.array_equal(rt.idx.cpu().numpy(), o_idx)
    assert np.all(np.abs(rt.w.cpu().numpy().astype(np.float64) - o_w) <= 1e-6 * o_w)
    exact = np.arange(cfg.T)
    OL = oracle.Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2,
                      R_up=Ru, R_down=Rd)
    _, Y64 = OL.forward(X, o_idx, o_w)
    ob = OL.backward(X, dY, o_idx, o_w)
    assert_close(bits_to_f64(t2np_bits(Y))[exact], Y64[exact], "tiny Y")
    assert_close(bits_to_f64(t2np_bits(dX))[exact], ob["dX64"][exact], "tiny dX")


def test_full_tiles_and_chunked_k_are_deterministic():
    """Token tiles up to the full 256 rows and a gate/up contraction long
    enough for the chunked accumulation (d = 4096: 64 K steps): four forwards
    with chunk sizes 2, 4, 16 and 4 again give bit-identical Y, and the
    saved g | u, h and h~ are identical too."""
    cfg = gi.LayerConfig("m", T=768, d=4096, E=16, k=8, I=512, b=64, C=4, seed=9)
    c = make_case(cfg, skew=0.5)
    L = DeviceLayer(cfg, c["w13"], c["s13"], c["w2"], c["s2"], R_up=c["R_up"], R_down=c["R_down"])
    rt = L.new_routing()
    rt.idx.copy_(torch.from_numpy(c["idx"]))
    rt.w.copy_(torch.from_numpy(c["w"]))
    L.permute(rt)
    assert int(rt.counts.max()) > 256            # some experts span several full tiles
    X = dev(c["X"])
    outs = []
    for C in (2, 4, 16, 4):
        Y = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device="cuda")
        ctx = L.new_ctx()
        L.forward(X, rt, Y, C=C, ctx=ctx)
        torch.cuda.synchronize()
        outs.append((t2np_bits(Y), ctx.cpu().numpy()))
    assert L.status() == pmoe.PMOE_OK
    for Y, ctx in outs[1:]:
        assert np.array_equal(Y, outs[0][0])
        assert np.array_equal(ctx, outs[0][1])


def test_dropped_pair_gets_zero_routing_gradient():
    """An expert id outside [0, E) leaves its pair out of the grouping (the
    permute reports PMOE_ERR_BAD_INDEX); the backward still runs, writes
    d_topk_w = 0 for that pair and finite values everywhere else, and writes
    nothing out of bounds."""
    cfg = gi.CONFIGS["tiny"]
    c = make_case(cfg)
    idx = c["idx"].copy()
    idx[5, 1] = cfg.E                       # out of range
    L = DeviceLayer(cfg, c["w13"], c["s13"], c["w2"], c["s2"], R_up=c["R_up"], R_down=c["R_down"])
    rt = L.new_routing()
    rt.idx.copy_(torch.from_numpy(idx))
    rt.w.copy_(torch.from_numpy(c["w"]))
    L.permute(rt)
    assert int(rt.offsets[cfg.E]) == cfg.P - 1
    X = dev(c["X"])
    Y = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device="cuda")
    ctx = L.new_ctx()
    L.forward(X, rt, Y, ctx=ctx)
    dX = torch.empty_like(Y)
    dtw = torch.full((cfg.T, cfg.k), float("nan"), dtype=torch.float32, device="cuda")
    dRu, dRd = L.grads()
    L.backward(X, dev(c["dY"]), ctx, rt, dX, dtw, dRu, dRd)
    torch.cuda.synchronize()
    assert L.status() == pmoe.PMOE_ERR_BAD_INDEX
    d = dtw.cpu().numpy()
    assert d[5, 1] == 0.0
    assert np.all(np.isfinite(d))
    assert np.all(np.isfinite(bits_to_f64(t2np_bits(dX))))
