"""Pins of the oracle's router, grouping, adapter, Cayley map, forward and
backward-data against facts other than the oracle itself: library routines
(numpy matmul / argsort / inv, scipy softmax), closed forms, invariants,
exact special cases and central finite differences."""
import numpy as np
import pytest
import scipy.special

import oracle
from precision_moe_adapter_gb300 import inputs as gi


def bf(h):
    return gi.bf16_bits_to_f32(h).astype(np.float64)


# ---------------------------------------------------------------- router

def test_route_logits_topk_softmax():
    cfg = gi.LayerConfig("r", T=40, d=64, E=16, k=4, I=32, b=16, router="zipf")
    X = gi.gen_x(cfg)
    Wr, bias = gi.gen_router(cfg)
    logits, idx, w = oracle.route(X, Wr, bias, cfg.k)
    ref = (bf(X) @ Wr.astype(np.float64) + bias.astype(np.float64)).astype(np.float32)
    assert np.max(np.abs(logits - ref) / np.spacing(np.abs(ref))) <= 1.0
    for t in range(cfg.T):
        order = np.lexsort((np.arange(cfg.E), -logits[t].astype(np.float64)))
        assert list(idx[t]) == list(order[:cfg.k])
        sel = logits[t][idx[t]].astype(np.float64)
        assert abs(w[t].astype(np.float64).sum() - 1) < 1e-6
        assert np.all(np.diff(w[t]) <= 0)
        ratio = w[t][1:].astype(np.float64) / w[t][0]
        assert np.allclose(ratio, np.exp(sel[1:] - sel[0]), rtol=1e-6)


def test_route_full_softmax_and_ties():
    cfg = gi.LayerConfig("r", T=8, d=32, E=6, k=6, I=32, b=16)
    X = gi.gen_x(cfg)
    Wr, _ = gi.gen_router(cfg)
    Wr[:, 4] = Wr[:, 1]                       # experts 1 and 4 always tie
    logits, idx, w = oracle.route(X, Wr, None, cfg.k)
    for t in range(cfg.T):
        pos = list(idx[t])
        assert pos.index(1) < pos.index(4)    # tie -> lower id first
        want = scipy.special.softmax(logits[t].astype(np.float64))[idx[t]]
        assert np.allclose(w[t], want, rtol=1e-6, atol=1e-9)


def test_topk_against_lexsort_and_softmax():
    """or_topk on given logits: the order of numpy's lexsort by (logit
    descending, id ascending), weights equal to scipy's softmax over the k
    selected (rounded to FP32); planted ties go to the lower id."""
    rng = np.random.default_rng(3)
    T, E, k = 200, 37, 7
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 20] = logits[:, 3]             # ties between experts 3 and 20
    logits[::3, 11] = logits[::3].max(axis=1)  # ties for the first slot
    idx, w = oracle.topk(logits, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))[:k]
        assert list(idx[t]) == list(order)
        want = scipy.special.softmax(logits[t][order].astype(np.float64)).astype(np.float32)
        assert np.allclose(w[t], want, rtol=2.5e-7, atol=0)


def test_route_canonical_order():
    """The canonical-order logits: (a) within the FP32 summation bound of
    the exact logits; (b) d = 32: each partial is one rounded product, and
    the tree s[i] += s[i + h] (h = 16 .. 1) reproduced with numpy float32
    additions gives the same bits; (c) with inputs whose products and
    partial sums are exact in FP32 the result is the exact dot product
    (no term dropped or counted twice)."""
    cfg = gi.LayerConfig("r", T=24, d=256, E=12, k=2, I=32, b=16, router="zipf")
    X = gi.gen_x(cfg)
    Wr, bias = gi.gen_router(cfg)
    lc = oracle.route_canonical(X, Wr, bias)
    x, W = bf(X), Wr.astype(np.float64)
    exact = x @ W + bias.astype(np.float64)
    bound = (cfg.d / 32 + 6) * 2.0 ** -24 * (np.abs(x) @ np.abs(W) + np.abs(bias))
    assert np.all(np.abs(lc - exact) <= bound)
    # (b) d = 32
    X32, W32 = X[:, :32], np.ascontiguousarray(Wr[:32])
    l32 = oracle.route_canonical(X32, W32, None)
    prod = (bf(X32)[:, :, None] * W32.astype(np.float64)[None]).astype(np.float32)   # [T, 32, E]
    s = prod.copy()
    for h in (16, 8, 4, 2, 1):
        s[:, :h] = (s[:, :h] + s[:, h:2 * h]).astype(np.float32)
    assert np.array_equal(l32, s[:, 0])
    # (c) small integers times eighths: every step exact in FP32
    rng = np.random.default_rng(4)
    Xi = gi.f32_to_bf16_bits(rng.integers(-8, 9, size=(9, 160)).astype(np.float32))
    Wi = (rng.integers(-8, 9, size=(160, 5)) / 8.0).astype(np.float32)
    li = oracle.route_canonical(Xi, Wi, None)
    assert np.array_equal(li.astype(np.float64), bf(Xi) @ Wi.astype(np.float64))


# ---------------------------------------------------------------- permute

@pytest.mark.parametrize("T,E,k", [(50, 8, 2), (1, 16, 8), (0, 4, 2), (37, 64, 6)])
def test_permute_against_stable_argsort(T, E, k):
    cfg = gi.LayerConfig("p", T=T, d=32, E=E, k=k, I=32, b=16)
    idx, _ = gi.gen_routing(cfg) if T else (np.zeros((0, k), np.int32), None)
    r = oracle.permute(idx, E)
    flat = idx.ravel()
    P = flat.size
    assert np.array_equal(r["counts"], np.bincount(flat, minlength=E))
    assert r["counts"].sum() == T * k and r["offsets"][E] == P
    assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(r["counts"])]))
    assert np.array_equal(r["perm"], np.argsort(flat, kind="stable"))
    assert np.array_equal(r["inv_perm"][r["perm"]], np.arange(P))
    act = np.flatnonzero(r["counts"])
    assert r["num_active"] == len(act)
    assert np.array_equal(r["active"][:len(act)], act) and np.all(r["active"][len(act):] == -1)


# ---------------------------------------------------------------- Cayley

def test_cayley_closed_form_b2():
    a = np.array([0.0, 0.3, -1.7, 5.0])
    S = np.zeros((4, 2, 2))
    S[:, 0, 1], S[:, 1, 0] = a, -a
    R = oracle.cayley(S)
    want = np.stack([np.array([[1 - x * x, 2 * x], [-2 * x, 1 - x * x]]) / (1 + x * x) for x in a])
    assert np.allclose(R, want, atol=1e-15)


@pytest.mark.parametrize("b", [16, 32, 64])
def test_cayley_orthogonal_and_library(b):
    S = gi.gen_skew(1, 4 * b, b, seed=5, sid="S_up", std=0.3)[0].astype(np.float64)
    R = oracle.cayley(S)
    I = np.eye(b)
    for blk in range(S.shape[0]):
        Rb = R[blk]
        assert np.max(np.abs(Rb.T @ Rb - I)) < 1e-12
        assert abs(np.linalg.det(Rb) - 1) < 1e-10
        assert np.allclose(Rb, (I + S[blk]) @ np.linalg.inv(I - S[blk]), atol=1e-12)
    assert np.array_equal(oracle.cayley(np.zeros((2, b, b))), np.broadcast_to(I, (2, b, b)))


def test_cayley_grad_finite_differences():
    b = 8
    S = gi.gen_skew(1, 2 * b, b, seed=6, sid="S_up", std=0.2)[0].astype(np.float64)
    G = np.random.default_rng(7).standard_normal(S.shape)
    dS = oracle.cayley_grad(S, G)
    assert np.allclose(dS, -np.swapaxes(dS, -1, -2))
    h = 1e-6
    for blk in range(S.shape[0]):
        for i in range(b):
            for j in range(i + 1, b):
                Sp, Sm = S.copy(), S.copy()
                Sp[blk, i, j] += h; Sp[blk, j, i] -= h
                Sm[blk, i, j] -= h; Sm[blk, j, i] += h
                fd = (np.sum(G * oracle.cayley(Sp)) - np.sum(G * oracle.cayley(Sm))) / (2 * h)
                assert abs(fd - dS[blk, i, j]) < 1e-6 * (1 + abs(fd))


# ---------------------------------------------------------------- adapter

def _blockdiag(R):
    nb, b, _ = R.shape
    M = np.zeros((nb * b, nb * b))
    for i in range(nb):
        M[i * b:(i + 1) * b, i * b:(i + 1) * b] = R[i]
    return M


def test_adapter_apply_and_grad_against_numpy():
    rows, dim, b = 33, 96, 32
    rng = np.random.default_rng(8)
    X = gi.f32_to_bf16_bits(rng.standard_normal((rows, dim)).astype(np.float32))
    dXr = gi.f32_to_bf16_bits(rng.standard_normal((rows, dim)).astype(np.float32))
    S = gi.gen_skew(1, dim, b, seed=9, sid="S_up", std=0.1)[0].astype(np.float64)
    Rb = gi.f32_to_bf16_bits(oracle.cayley(S).astype(np.float32))
    M = _blockdiag(bf(Rb))
    got = oracle.adapter_apply(X, Rb, b)
    assert np.array_equal(got, oracle.bf16_round(bf(X) @ M).reshape(rows, dim))
    dX, dR = oracle.adapter_grad(X, dXr, Rb, b)
    assert np.array_equal(dX, oracle.bf16_round(bf(dXr) @ M.T).reshape(rows, dim))
    want = np.einsum("ibr,ibc->brc", bf(X).reshape(rows, dim // b, b), bf(dXr).reshape(rows, dim // b, b))
    assert np.allclose(dR, want, rtol=1e-12, atol=1e-12)


def test_adapter_apply_permutation_is_exact():
    rows, dim, b = 5, 64, 16
    X = gi.gen_x(gi.LayerConfig("a", T=rows, d=dim, E=1, k=1, I=32, b=b))
    rng = np.random.default_rng(10)
    R = np.zeros((dim // b, b, b))
    for i in range(dim // b):
        R[i][np.arange(b), rng.permutation(b)] = 1.0
    Rb = gi.f32_to_bf16_bits(R.astype(np.float32))
    got = oracle.adapter_apply(X, Rb, b)
    assert np.array_equal(bf(got), bf(X) @ _blockdiag(R))


# ---------------------------------------------------------------- layer

def _small(fmt=gi.INT4, T=6, d=64, E=4, k=2, I=64, b=16, adapter="per_expert", seed=0):
    cfg = gi.LayerConfig("s", T=T, d=d, E=E, k=k, I=I, b=b, fmt=fmt, adapter=adapter, seed=seed)
    w13, s13, w2, s2 = gi.gen_weights(cfg)
    return cfg, (w13, s13, w2, s2)


def _dense(fmt, q, s, N, K):
    return bf(oracle.dequant(fmt, q, s, N, K))


@pytest.mark.parametrize("fmt", [gi.INT4, gi.MXFP4])
def test_forward_single_expert_is_textbook_swiglu(fmt):
    """E = 1, k = 1, no adapter, no rounding: a dense SwiGLU MLP."""
    cfg, (w13, s13, w2, s2) = _small(fmt, E=1, k=1)
    X = gi.gen_x(cfg)
    L = oracle.Layer(cfg.T, cfg.d, 1, 1, cfg.I, cfg.b, fmt, w13, s13, w2, s2)
    idx = np.zeros((cfg.T, 1), np.int32)
    w = np.ones((cfg.T, 1), np.float32)
    _, Y64 = L.forward(X, idx, w, no_round=True)
    W13 = _dense(fmt, w13[0], s13[0], 2 * cfg.I, cfg.d)
    W2 = _dense(fmt, w2[0], s2[0], cfg.d, cfg.I)
    x = bf(X)
    g, u = x @ W13[:cfg.I].T, x @ W13[cfg.I:].T
    want = (g / (1 + np.exp(-g)) * u) @ W2.T
    assert np.allclose(Y64, want, rtol=1e-12, atol=1e-12)


def test_forward_fp8_single_expert_textbook():
    cfg, (w13, s13, w2, s2) = _small(gi.FP8, E=1, k=1, d=256, I=128, T=3)
    X = gi.gen_x(cfg)
    L = oracle.Layer(cfg.T, cfg.d, 1, 1, cfg.I, cfg.b, gi.FP8, w13, s13, w2, s2)
    _, Y64 = L.forward(X, np.zeros((3, 1), np.int32), np.ones((3, 1), np.float32), no_round=True)
    W13 = _dense(gi.FP8, w13[0], s13[0], 2 * cfg.I, cfg.d)
    W2 = _dense(gi.FP8, w2[0], s2[0], cfg.d, cfg.I)
    x = bf(X)
    g, u = x @ W13[:cfg.I].T, x @ W13[cfg.I:].T
    assert np.allclose(Y64, (g / (1 + np.exp(-g)) * u) @ W2.T, rtol=1e-12, atol=1e-12)


def test_forward_rotations_side_and_orientation():
    """Permutation blocks are exact in BF16, so with rounding on, rotating
    by R_up = P equals feeding X P to the adapter-less layer, and R_down = Q
    equals (silu(g) u) Q before the down projection (no-round textbook)."""
    cfg, (w13, s13, w2, s2) = _small(E=1, k=1)
    X = gi.gen_x(cfg)
    rng = np.random.default_rng(11)

    def perm_blocks(dim):
        R = np.zeros((dim // cfg.b, cfg.b, cfg.b))
        for i in range(dim // cfg.b):
            R[i][np.arange(cfg.b), rng.permutation(cfg.b)] = 1.0
        return R

    Pu, Qd = perm_blocks(cfg.d), perm_blocks(cfg.I)
    bits = lambda R: gi.f32_to_bf16_bits(R.astype(np.float32))[None]
    idx, w = np.zeros((cfg.T, 1), np.int32), np.ones((cfg.T, 1), np.float32)
    base = oracle.Layer(cfg.T, cfg.d, 1, 1, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2)
    rot = oracle.Layer(cfg.T, cfg.d, 1, 1, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2, R_up=bits(Pu))
    XP = gi.f32_to_bf16_bits((bf(X) @ _blockdiag(Pu)).astype(np.float32))
    assert np.array_equal(rot.forward(X, idx, w)[0], base.forward(XP, idx, w)[0])
    rot2 = oracle.Layer(cfg.T, cfg.d, 1, 1, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2, R_down=bits(Qd))
    _, Y64 = rot2.forward(X, idx, w, no_round=True)
    W13 = _dense(cfg.fmt, w13[0], s13[0], 2 * cfg.I, cfg.d)
    W2 = _dense(cfg.fmt, w2[0], s2[0], cfg.d, cfg.I)
    g, u = bf(X) @ W13[:cfg.I].T, bf(X) @ W13[cfg.I:].T
    want = ((g / (1 + np.exp(-g)) * u) @ _blockdiag(Qd)) @ W2.T
    assert np.allclose(Y64, want, rtol=1e-12, atol=1e-12)


def test_zero_adapter_is_the_base_bit_exact():
    """The reference policy is the adapter disabled; S = 0 gives R = I and
    must reproduce the adapter-less layer exactly."""
    cfg, (w13, s13, w2, s2) = _small()
    X = gi.gen_x(cfg)
    idx, w = gi.gen_routing(cfg)
    nu, nd = cfg.d // cfg.b, cfg.I // cfg.b
    Ru = gi.f32_to_bf16_bits(oracle.cayley(np.zeros((cfg.E * nu, cfg.b, cfg.b))).astype(np.float32))
    Rd = gi.f32_to_bf16_bits(oracle.cayley(np.zeros((cfg.E * nd, cfg.b, cfg.b))).astype(np.float32))
    off = oracle.Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2)
    on = oracle.Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2,
                      R_up=Ru.reshape(cfg.E, nu, cfg.b, cfg.b), R_down=Rd.reshape(cfg.E, nd, cfg.b, cfg.b))
    Y0, Y064 = off.forward(X, idx, w)
    Y1, Y164 = on.forward(X, idx, w)
    assert np.array_equal(Y0, Y1) and np.array_equal(Y064, Y164)


def test_forward_is_weighted_sum_of_experts():
    cfg, (w13, s13, w2, s2) = _small(E=5, k=3)
    X = gi.gen_x(cfg)
    idx, w = gi.gen_routing(cfg)
    L = oracle.Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2)
    Y, Y64, o = L.forward(X, idx, w, want_o=True)
    L1 = oracle.Layer(cfg.T, cfg.d, cfg.E, 1, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2)
    acc = np.zeros_like(Y64)
    for j in range(cfg.k):
        _, Yj = L1.forward(X, idx[:, j:j + 1], np.ones((cfg.T, 1), np.float32))
        acc += w[:, j:j + 1].astype(np.float64) * Yj
        assert np.array_equal(Yj, o.reshape(cfg.T, cfg.k, cfg.d)[:, j])
    assert np.allclose(Y64, acc, rtol=1e-14, atol=1e-14)
    assert np.array_equal(Y, oracle.bf16_round(Y64).reshape(Y.shape))
    # a token subset computes the same rows
    Ys, _ = L.forward(X, idx, w, toks=[4, 1])
    assert np.array_equal(Ys[[1, 4]], Y[[1, 4]]) and not Ys[0].any()


def _fd_layer(adapter="per_expert"):
    cfg, (w13, s13, w2, s2) = _small(T=3, d=32, E=3, k=2, I=32, b=16, adapter=adapter)
    X64 = np.random.default_rng(12).standard_normal((cfg.T, cfg.d))
    dY = gi.gen_dy(cfg)
    idx, w = gi.gen_routing(cfg)
    n = 1 if adapter == "shared" else cfg.E
    Su, Sd = gi.gen_skew(n, cfg.d, cfg.b, 0, "S_up", 0.2), gi.gen_skew(n, cfg.I, cfg.b, 0, "S_down", 0.2)
    Ru = oracle.cayley(Su.reshape(-1, cfg.b, cfg.b)).reshape(Su.shape)
    Rd = oracle.cayley(Sd.reshape(-1, cfg.b, cfg.b)).reshape(Sd.shape)
    mk = lambda ru, rd: oracle.Layer(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b, cfg.fmt, w13, s13,
                                     w2, s2, R_up64=ru, R_down64=rd)
    return cfg, mk, X64, dY, idx, w, Ru, Rd


@pytest.mark.parametrize("adapter", ["per_expert", "shared"])
def test_backward_finite_differences(adapter):
    cfg, mk, X64, dY, idx, w, Ru, Rd = _fd_layer(adapter)
    L = mk(Ru, Rd)
    g = L.backward(None, dY, idx, w, no_round=True, X64=X64)
    dy = bf(dY)
    loss = lambda lay, x: float(np.sum(dy * lay.forward(None, idx, w, no_round=True, X64=x)[1]))
    h = 1e-5
    rng = np.random.default_rng(13)
    for _ in range(12):
        t, c = rng.integers(cfg.T), rng.integers(cfg.d)
        Xp, Xm = X64.copy(), X64.copy()
        Xp[t, c] += h; Xm[t, c] -= h
        fd = (loss(L, Xp) - loss(L, Xm)) / (2 * h)
        assert abs(fd - g["dX64"][t, c]) < 1e-7 * (1 + abs(fd))
    for name, R, which in (("dR_up", Ru, 0), ("dR_down", Rd, 1)):
        for _ in range(12):
            pos = tuple(rng.integers(s) for s in R.shape)
            Rp, Rm = R.copy(), R.copy()
            Rp[pos] += h; Rm[pos] -= h
            Lp = mk(Rp, Rd) if which == 0 else mk(Ru, Rp)
            Lm = mk(Rm, Rd) if which == 0 else mk(Ru, Rm)
            fd = (loss(Lp, X64) - loss(Lm, X64)) / (2 * h)
            assert abs(fd - g[name][pos]) < 1e-7 * (1 + abs(fd)), (name, pos)
    # d_topk_w[t, j] = dY_t . o_j (Y is linear in the routing weights)
    _, _, o = L.forward(None, idx, w, no_round=True, want_o=True, X64=X64)
    want = np.einsum("tc,tjc->tj", dy, o.reshape(cfg.T, cfg.k, cfg.d))
    assert np.allclose(g["d_topk_w"], want, rtol=1e-6, atol=1e-9)


def test_backward_rounded_close_to_exact():
    """With the BF16 rounding points on, the gradients stay within BF16
    error of the exact ones (sanity of the rounding placement)."""
    cfg, mk, X64, dY, idx, w, Ru, Rd = _fd_layer()
    Xb = gi.f32_to_bf16_bits(X64.astype(np.float32))
    L = mk(Ru, Rd)
    ex = L.backward(None, dY, idx, w, no_round=True, X64=bf(Xb))
    rd = L.backward(None, dY, idx, w, no_round=False, X64=bf(Xb))
    rel = np.linalg.norm(rd["dX64"] - ex["dX64"]) / np.linalg.norm(ex["dX64"])
    assert rel < 2e-2
    assert np.array_equal(rd["dX"], oracle.bf16_round(rd["dX64"]).reshape(rd["dX"].shape))


def test_forward_rounding_points_against_torch():
    """BF16 rounding of x~, h and h~ (and Y), checked against a torch
    computation that rounds with torch's own conversions."""
    import torch
    cfg, (w13, s13, w2, s2) = _small(E=1, k=1, T=5)
    X = gi.gen_x(cfg)
    Su = gi.gen_skew(1, cfg.d, cfg.b, 0, "S_up", 0.05)
    Sd = gi.gen_skew(1, cfg.I, cfg.b, 0, "S_down", 0.05)
    Ru = gi.f32_to_bf16_bits(oracle.cayley(Su.reshape(-1, cfg.b, cfg.b)).astype(np.float32)).reshape(Su.shape)
    Rd = gi.f32_to_bf16_bits(oracle.cayley(Sd.reshape(-1, cfg.b, cfg.b)).astype(np.float32)).reshape(Sd.shape)
    L = oracle.Layer(cfg.T, cfg.d, 1, 1, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2, R_up=Ru, R_down=Rd)
    idx, w = np.zeros((cfg.T, 1), np.int32), np.ones((cfg.T, 1), np.float32)
    Y, Y64 = L.forward(X, idx, w)
    r = lambda a: torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    W13 = _dense(cfg.fmt, w13[0], s13[0], 2 * cfg.I, cfg.d)
    W2 = _dense(cfg.fmt, w2[0], s2[0], cfg.d, cfg.I)
    xt = r(bf(X) @ _blockdiag(bf(Ru[0])))
    g, u = xt @ W13[:cfg.I].T, xt @ W13[cfg.I:].T
    h = r(g / (1 + np.exp(-g)) * u)
    ht = r(h @ _blockdiag(bf(Rd[0])))
    want = ht @ W2.T                 # each pair's output o keeps its precision
    assert np.allclose(Y64, want, rtol=1e-12, atol=1e-12)
    assert np.array_equal(bf(Y), r(want))
    # the values the two down-path decisions are taken on
    hx = L.pre_round(X, idx, np.arange(cfg.T))
    assert np.allclose(hx[:, :cfg.I], g / (1 + np.exp(-g)) * u, rtol=1e-12, atol=1e-12)
    assert np.allclose(hx[:, cfg.I:], h @ _blockdiag(bf(Rd[0])), rtol=1e-12, atol=1e-12)


def test_backward_rounding_points_against_torch():
    """The backward's only BF16 rounding points are those of the recomputed
    forward (x~, h, h~) and dX; g, u, dh~, dg, du, dx~ and the rotated dx
    keep their precision.  Checked against a torch-rounded computation (one
    expert, k = 1, a routing weight other than one)."""
    import torch
    cfg, (w13, s13, w2, s2) = _small(E=1, k=1, T=4)
    X, dY = gi.gen_x(cfg), gi.gen_dy(cfg)
    Su = gi.gen_skew(1, cfg.d, cfg.b, 0, "S_up", 0.05)
    Sd = gi.gen_skew(1, cfg.I, cfg.b, 0, "S_down", 0.05)
    rb = lambda S: gi.f32_to_bf16_bits(oracle.cayley(S.reshape(-1, cfg.b, cfg.b)).astype(np.float32)).reshape(S.shape)
    Ru, Rd = rb(Su), rb(Sd)
    L = oracle.Layer(cfg.T, cfg.d, 1, 1, cfg.I, cfg.b, cfg.fmt, w13, s13, w2, s2, R_up=Ru, R_down=Rd)
    idx, w = np.zeros((cfg.T, 1), np.int32), np.full((cfg.T, 1), 0.75, np.float32)
    ob = L.backward(X, dY, idx, w)
    r = lambda a: torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    W13 = _dense(cfg.fmt, w13[0], s13[0], 2 * cfg.I, cfg.d)
    Wg, Wu = W13[:cfg.I], W13[cfg.I:]
    W2 = _dense(cfg.fmt, w2[0], s2[0], cfg.d, cfg.I)
    BU, BD = _blockdiag(bf(Ru[0])), _blockdiag(bf(Rd[0]))
    x = bf(X)
    xt = r(x @ BU)
    g, u = xt @ Wg.T, xt @ Wu.T
    h = r(g / (1 + np.exp(-g)) * u)
    ht = r(h @ BD)
    G = bf(dY) @ W2
    dht = 0.75 * G
    dh = dht @ BD.T
    sg = 1 / (1 + np.exp(-g))
    dg = dh * u * sg * (1 + g * (1 - sg))
    du = dh * (g / (1 + np.exp(-g)))
    dxt = dg @ Wg + du @ Wu
    dxp = dxt @ BU.T
    assert np.allclose(ob["dX64"], dxp, rtol=1e-12, atol=1e-12)
    assert np.array_equal(bf(ob["dX"]), r(dxp))
    assert np.allclose(ob["d_topk_w"][:, 0], np.sum(G * ht, axis=1), rtol=1e-6)
    nb = lambda a: a.reshape(cfg.T, -1, cfg.b)
    assert np.allclose(ob["dR_up"][0], np.einsum("tbr,tbc->brc", nb(x), nb(dxt)), rtol=1e-12, atol=1e-12)
    assert np.allclose(ob["dR_down"][0], np.einsum("tbr,tbc->brc", nb(h), nb(dht)), rtol=1e-12, atol=1e-12)
