"""GPU parity of the single-step entry points against the oracle:
dequantization (bit-exact), grouping (bit-exact), router (logits within
the FP32 accumulation bound, selections exact where unique), adapter
rotation and gradient, Cayley map and its gradient."""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_adapter_gb300 import build, pmoe
from precision_moe_adapter_gb300 import inputs as gi
from helpers import assert_close, bits_to_f64, check_cayley, check_routing, check_topk, t2np_bits

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


# ---------------------------------------------------------------- dequant

def _all_finite_bf16_bits():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    return bits[np.isfinite(f)]


def _gpu_dequant(fmt, q, s, N, K):
    out = torch.empty((N, K), dtype=torch.int16, device="cuda")
    pmoe.moe_dequant(fmt, dev(q), dev(s), N, K, out)
    torch.cuda.synchronize()
    return t2np_bits(out)


def test_dequant_int4_exhaustive():
    sb = _all_finite_bf16_bits()
    N, K = len(sb), 32
    qv = np.tile(np.arange(16, dtype=np.uint8), 2)
    q = np.tile((qv[0::2] | (qv[1::2] << 4)).astype(np.uint8), (N, 1))
    s = sb.reshape(N, 1)
    assert np.array_equal(_gpu_dequant(0, q, s, N, K), oracle.dequant(0, q, s, N, K))


def test_dequant_mxfp4_exhaustive():
    N, K = 256, 32
    qv = np.tile(np.arange(16, dtype=np.uint8), 2)
    q = np.tile((qv[0::2] | (qv[1::2] << 4)).astype(np.uint8), (N, 1))
    s = np.arange(256, dtype=np.uint8).reshape(N, 1)
    got, want = _gpu_dequant(1, q, s, N, K), oracle.dequant(1, q, s, N, K)
    assert np.array_equal(got[:255], want[:255])
    assert np.all((got[255] & 0x7F80) == 0x7F80) and np.all(got[255] & 0x7F)   # NaN scale


def test_dequant_fp8_all_codes_many_scales():
    rng = np.random.default_rng(5)
    nb = 64
    sc = (rng.random((nb, 2)) * 0.015 + 0.005).astype(np.float32)
    sc[:8] = (rng.standard_normal((8, 2)) * 10.0 ** rng.integers(-30, 30, (8, 2))).astype(np.float32)
    N, K = 128 * nb, 256
    q = np.tile(np.arange(256, dtype=np.uint8), (N, 1))
    got, want = _gpu_dequant(2, q, sc, N, K), oracle.dequant(2, q, sc, N, K)
    nan = np.isnan(bits_to_f64(want))
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7F80) == 0x7F80)


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_dequant_random_matrices(fmt):
    N, K = 384, 512
    q, s = gi.gen_matrix(fmt, 1, N, K, seed=3, qsid="w13", ssid="s13")
    q, s = q[0], s[0]
    assert np.array_equal(_gpu_dequant(fmt, q, s, N, K), oracle.dequant(fmt, q, s, N, K))


# ---------------------------------------------------------------- permute

def _gpu_permute(idx, E):
    T, k = idx.shape
    dm = pmoe.dims(T, 64, E, k, 64, 16)
    i32 = dict(dtype=torch.int32, device="cuda")
    P = T * k
    bufs = dict(counts=torch.zeros(E, **i32), offsets=torch.zeros(E + 1, **i32),
                perm=torch.zeros(max(P, 1), **i32), inv_perm=torch.zeros(max(P, 1), **i32),
                active=torch.zeros(E, **i32), num_active=torch.zeros(1, **i32))
    rt = pmoe.routing(None, None, bufs["counts"], bufs["offsets"], bufs["perm"], bufs["inv_perm"],
                      bufs["active"], bufs["num_active"])
    ws = torch.zeros(max(pmoe.moe_workspace_bytes(dm, pmoe.OP_PERMUTE), 256), dtype=torch.uint8,
                     device="cuda")
    idx_d = dev(idx.astype(np.int32)) if P else torch.zeros(1, **i32)
    pmoe.moe_permute(dm, idx_d, rt, ws)
    st = pmoe.moe_query_status(ws)
    out = {k_: v.cpu().numpy() for k_, v in bufs.items()}
    out["perm"], out["inv_perm"] = out["perm"][:P], out["inv_perm"][:P]
    out["num_active"] = int(out["num_active"][0])
    return out, st


@pytest.mark.parametrize("T,E,k,skew", [(64, 8, 2, 1.1), (4096, 128, 8, 0.0), (8192, 384, 8, 1.1),
                                        (1, 384, 8, 1.1), (3000, 256, 8, 3.0), (777, 4096, 32, 1.1),
                                        (2048, 1, 1, 0.0)])
def test_permute_bit_exact(T, E, k, skew):
    cfg = gi.LayerConfig("p", T=T, d=64, E=E, k=k, I=64, b=16, seed=T + E)
    idx, _ = gi.gen_routing(cfg, skew=skew)
    got, st = _gpu_permute(idx, E)
    want = oracle.permute(idx, E)
    assert st == pmoe.PMOE_OK
    for key in ("counts", "offsets", "perm", "inv_perm", "active"):
        assert np.array_equal(got[key], want[key]), key
    assert got["num_active"] == want["num_active"]


def test_permute_empty_and_bad_index():
    got, st = _gpu_permute(np.zeros((0, 2), np.int32), 8)
    assert st == pmoe.PMOE_OK and got["num_active"] == 0 and not got["counts"].any()
    assert np.all(got["active"] == -1) and not got["offsets"].any()
    idx = np.array([[0, 1], [2, 9], [3, -1]], np.int32)
    got, st = _gpu_permute(idx, 8)
    assert st == pmoe.PMOE_ERR_BAD_INDEX
    assert got["counts"].sum() == 4 and got["offsets"][8] == 4
    assert got["inv_perm"][3] == -1 and got["inv_perm"][5] == -1


# ---------------------------------------------------------------- router

def _gpu_route(cfg, X, Wr, bias, mode=pmoe.ROUTE_FAST):
    dm = pmoe.dims(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b)
    ws = torch.zeros(pmoe.moe_workspace_bytes(dm, pmoe.OP_PERMUTE), dtype=torch.uint8, device="cuda")
    logits = torch.zeros((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    idx = torch.zeros((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.zeros((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    pmoe.moe_route(dm, dev(X), dev(Wr), None if bias is None else dev(bias), logits, idx, w, ws,
                   mode=mode)
    torch.cuda.synchronize()
    return logits.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("name,T", [("tiny", None), ("qwen3_30b_a3b", 256), ("kimi_k2", 96)])
def test_route_against_oracle(name, T):
    """Fast mode: logits within the FP32 bound, selection and weights
    bit-exact against the oracle's top-k on the device's logits, and every
    token routed differently from the oracle's own FP64 routing a
    certified near-tie (check_routing)."""
    cfg = gi.CONFIGS[name]
    if T:
        cfg = cfg.with_(T=T)
    X = gi.gen_x(cfg)
    Wr, bias = gi.gen_router(cfg)
    gl, gidx, gw = _gpu_route(cfg, X, Wr, bias)
    check_routing(X, Wr, bias, cfg.k, gl, gidx, gw)


@pytest.mark.parametrize("T,d,E,k,zipf", [(64, 256, 8, 2, False), (1, 64, 5, 3, True),
                                          (37, 192, 70, 8, True), (200, 2048, 128, 8, False),
                                          (96, 7168, 384, 8, True)])
def test_route_exact_mode_bit_exact(T, d, E, k, zipf):
    """Exact mode: the logits equal the oracle's canonical-order logits bit
    for bit, so the routing equals the oracle's (idx bit-exact, w within
    1e-6 relative) -- ragged expert counts, one token, the tiny and the
    Kimi-K2 router shapes."""
    cfg = gi.LayerConfig("rx", T=T, d=d, E=E, k=k, I=64, b=16, router="zipf" if zipf else "uniform")
    X = gi.gen_x(cfg)
    Wr, bias = gi.gen_router(cfg)
    gl, gidx, gw = _gpu_route(cfg, X, Wr, bias, mode=pmoe.ROUTE_EXACT)
    ol = oracle.route_canonical(X, Wr, bias)
    assert np.array_equal(gl.view(np.uint32), ol.view(np.uint32))
    check_topk(gl, gidx, gw, k)
    o_idx, o_w = oracle.topk(ol, k)
    assert np.array_equal(gidx, o_idx)


def test_route_ties_to_lower_id():
    cfg = gi.LayerConfig("t", T=32, d=64, E=16, k=4, I=64, b=16)
    X = gi.gen_x(cfg)
    Wr, _ = gi.gen_router(cfg)
    Wr[:, 9] = Wr[:, 2]
    Wr[:, 12] = Wr[:, 2]
    _, gidx, _ = _gpu_route(cfg, X, Wr, None)
    for t in range(cfg.T):
        s = list(gidx[t])
        pos = [s.index(e) if e in s else 99 for e in (2, 9, 12)]
        assert pos == sorted(pos)


# ---------------------------------------------------------------- adapter

@pytest.mark.parametrize("dim,b,rows", [(256, 32, 100), (7168, 64, 40), (2048, 64, 300), (512, 128, 33),
                                        (96, 16, 7)])
def test_adapter_apply_and_grad(dim, b, rows):
    rng = np.random.default_rng(dim + b)
    X = gi.f32_to_bf16_bits(rng.standard_normal((rows, dim)).astype(np.float32))
    dXr = gi.f32_to_bf16_bits(rng.standard_normal((rows, dim)).astype(np.float32))
    S = gi.gen_skew(1, dim, b, seed=1, sid="S_up", std=0.05)[0]
    R = gi.f32_to_bf16_bits(oracle.cayley(S).astype(np.float32))
    Xr = torch.empty((rows, dim), dtype=torch.int16, device="cuda")
    pmoe.adapter_apply(rows, dim, b, dev(X), dev(R), Xr)
    dX = torch.empty((rows, dim), dtype=torch.int16, device="cuda")
    dR = torch.empty((dim // b, b, b), dtype=torch.float32, device="cuda")
    pmoe.adapter_grad(rows, dim, b, dev(X), dev(dXr), dev(R), dX, dR)
    torch.cuda.synchronize()
    want = oracle.adapter_apply(X, R, b)
    got = t2np_bits(Xr)
    wdX, wdR = oracle.adapter_grad(X, dXr, R, b)
    if b <= 64:
        # BF16 outputs rounded as the exact sums are (near a rounding
        # midpoint the sum is recomputed error-free): bit-exact
        assert np.array_equal(got, want)
        assert np.array_equal(t2np_bits(dX), wdX)
    else:
        assert_close(bits_to_f64(got), bits_to_f64(want), "Xr", rel_fro=2e-3, max_abs=1e-2)
        assert np.mean(got == want) > 0.95
        assert_close(bits_to_f64(t2np_bits(dX)), bits_to_f64(wdX), "dX", rel_fro=2e-3, max_abs=1e-2)
    assert_close(dR.cpu().numpy(), wdR, "dR", rel_fro=1e-5, max_abs=1e-4)


@pytest.mark.parametrize("b,rows", [(64, 3001), (32, 517)])
def test_rotation_exact_at_all_magnitudes(b, rows):
    """x R and x R^T rounded to BF16 as the exact sums are, bit for bit,
    with rows spread over 2^-40 .. 2^40 so that many results sit near a
    rounding midpoint (those take the error-free recomputation)."""
    dim = 1024
    rng = np.random.default_rng(b * 7 + rows)
    z = rng.standard_normal((rows, dim)) * np.exp2(rng.integers(-40, 41, (rows, 1)))
    z[::7] *= np.exp2(rng.integers(-6, 7, (1, dim)))          # mixed magnitudes inside rows
    X = gi.f32_to_bf16_bits(z.astype(np.float32))
    S = gi.gen_skew(1, dim, b, seed=3, sid="S_up", std=0.02)[0]
    R = gi.f32_to_bf16_bits(oracle.cayley(S).astype(np.float32))
    Xr = torch.empty((rows, dim), dtype=torch.int16, device="cuda")
    pmoe.adapter_apply(rows, dim, b, dev(X), dev(R), Xr)
    dX = torch.empty((rows, dim), dtype=torch.int16, device="cuda")
    dR = torch.empty((dim // b, b, b), dtype=torch.float32, device="cuda")
    pmoe.adapter_grad(rows, dim, b, dev(X), dev(X), dev(R), dX, dR)
    torch.cuda.synchronize()
    assert np.array_equal(t2np_bits(Xr), oracle.adapter_apply(X, R, b))
    wdX, _ = oracle.adapter_grad(X, X, R, b)
    assert np.array_equal(t2np_bits(dX), wdX)


@pytest.mark.parametrize("b,std", [(2, 0.5), (16, 0.3), (32, 0.01), (64, 0.01), (128, 0.05)])
def test_cayley_and_grad(b, std):
    S = gi.gen_skew(3, 2 * b, b, seed=b, sid="S_up", std=std).reshape(-1, b, b)
    nblk = S.shape[0]
    Rb = torch.empty((nblk, b, b), dtype=torch.int16, device="cuda")
    Rf = torch.empty((nblk, b, b), dtype=torch.float32, device="cuda")
    pmoe.adapter_cayley(nblk, b, dev(S), Rb, Rf)
    G = np.random.default_rng(b).standard_normal((nblk, b, b)).astype(np.float32)
    dS = torch.empty((nblk, b, b), dtype=torch.float32, device="cuda")
    pmoe.adapter_cayley_grad(nblk, b, dev(S), Rf, dev(G), dS)
    torch.cuda.synchronize()
    R64 = oracle.cayley(S)
    rf = Rf.cpu().numpy()
    # FP32 elimination on b x b: error within a few b * 2^-24 (|A| <= 1)
    eps = 4 * b * 2.0 ** -24
    assert np.max(np.abs(rf - R64)) < eps
    for blk in range(nblk):
        assert np.max(np.abs(rf[blk].T.astype(np.float64) @ rf[blk] - np.eye(b))) < 4 * eps
    # R_bf16 = bf16(R_f32): equal to bf16 of the exact R except at certified
    # near-midpoints
    check_cayley(t2np_bits(Rb), rf, R64, b)
    want = oracle.cayley_grad(S, G)
    assert_close(dS.cpu().numpy(), want, "dS", rel_fro=1e-5, max_abs=1e-4)
