"""Pins of the oracle's dense bypass-base-weight-grad linear with the OFT
adapter (one frozen projection outside the experts): y = x~ W^T with
x~ = bf16(x blockdiag(R)); the backward gives dX and dR, no dW."""
import numpy as np
import pytest

import oracle
from precision_moe_adapter_gb300 import inputs as gi


def bf(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _blockdiag(R):
    n, b, _ = R.shape
    out = np.zeros((n * b, n * b))
    for i in range(n):
        out[i * b:(i + 1) * b, i * b:(i + 1) * b] = R[i]
    return out


def _case(fmt=gi.INT4, rows=5, N=128, K=128, b=32, seed=3):
    q, s = gi.gen_matrix(fmt, 1, N, K, seed=seed, qsid="w2", ssid="s2")
    X = gi.f32_to_bf16_bits(np.random.default_rng(seed).standard_normal((rows, K)).astype(np.float32))
    dY = gi.f32_to_bf16_bits(0.1 * np.random.default_rng(seed + 1).standard_normal((rows, N)).astype(np.float32))
    W = bf(oracle.dequant(fmt, q[0], s[0], N, K))
    return q[0], s[0], X, dY, W


@pytest.mark.parametrize("fmt", [gi.INT4, gi.MXFP4, gi.FP8])
def test_without_adapter_is_the_textbook_product(fmt):
    q, s, X, dY, W = _case(fmt)
    N, K = W.shape
    Y, Y64 = oracle.dense_forward(fmt, q, s, N, K, 32, None, X)
    assert np.allclose(Y64, bf(X) @ W.T, rtol=1e-12, atol=1e-12)
    assert np.array_equal(Y, oracle.bf16_round(Y64).reshape(Y.shape))
    g = oracle.dense_backward(fmt, q, s, N, K, 32, None, X, dY)
    assert g["dR"] is None
    assert np.allclose(g["dX64"], bf(dY) @ W, rtol=1e-12, atol=1e-12)


def test_rotation_side_with_exact_permutation_blocks():
    q, s, X, dY, W = _case()
    N, K = W.shape
    b = 32
    rng = np.random.default_rng(5)
    P = np.zeros((K // b, b, b))
    for i in range(K // b):
        P[i][np.arange(b), rng.permutation(b)] = 1.0
    Pb = gi.f32_to_bf16_bits(P.astype(np.float32))
    XP = gi.f32_to_bf16_bits((bf(X) @ _blockdiag(P)).astype(np.float32))
    assert np.array_equal(oracle.dense_forward(gi.INT4, q, s, N, K, b, Pb, X)[0],
                          oracle.dense_forward(gi.INT4, q, s, N, K, b, None, XP)[0])


def test_backward_finite_differences():
    q, s, X, dY, W = _case(rows=3, N=64, K=64, b=16)
    N, K, b = 64, 64, 16
    X64 = np.random.default_rng(9).standard_normal((3, K))
    S = gi.gen_skew(1, K, b, 0, "S_up", 0.2)[0]
    R = oracle.cayley(S)
    g = oracle.dense_backward(gi.INT4, q, s, N, K, b, None, None, dY, no_round=True, R64=R, X64=X64)
    dy = bf(dY)
    loss = lambda x, r: float(np.sum(dy * oracle.dense_forward(gi.INT4, q, s, N, K, b, None, None,
                                                                no_round=True, R64=r, X64=x)[1]))
    h = 1e-5
    rng = np.random.default_rng(10)
    for _ in range(10):
        i, c = rng.integers(3), rng.integers(K)
        Xp, Xm = X64.copy(), X64.copy()
        Xp[i, c] += h; Xm[i, c] -= h
        fd = (loss(Xp, R) - loss(Xm, R)) / (2 * h)
        assert abs(fd - g["dX64"][i, c]) < 1e-7 * (1 + abs(fd))
    for _ in range(10):
        pos = tuple(rng.integers(n) for n in R.shape)
        Rp, Rm = R.copy(), R.copy()
        Rp[pos] += h; Rm[pos] -= h
        fd = (loss(X64, Rp) - loss(X64, Rm)) / (2 * h)
        assert abs(fd - g["dR"][pos]) < 1e-7 * (1 + abs(fd))


def test_rounding_points_against_torch():
    """x~ and the outputs are BF16 tensors (torch's conversion); the
    backward's dx~ = dY W keeps its precision."""
    import torch
    q, s, X, dY, W = _case(rows=4)
    N, K, b = 128, 128, 32
    S = gi.gen_skew(1, K, b, 0, "S_up", 0.05)[0]
    Rb = gi.f32_to_bf16_bits(oracle.cayley(S).astype(np.float32))
    r = lambda a: torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    BD = _blockdiag(bf(Rb))
    xt = r(bf(X) @ BD)
    Y, Y64 = oracle.dense_forward(gi.INT4, q, s, N, K, b, Rb, X)
    assert np.allclose(Y64, xt @ W.T, rtol=1e-12, atol=1e-12)
    g = oracle.dense_backward(gi.INT4, q, s, N, K, b, Rb, X, dY)
    dxt = bf(dY) @ W
    assert np.allclose(g["dX64"], dxt @ BD.T, rtol=1e-12, atol=1e-12)
    assert np.array_equal(bf(g["dX"]), r(dxt @ BD.T))
    nb = lambda a: a.reshape(a.shape[0], -1, b)
    assert np.allclose(g["dR"], np.einsum("tbr,tbc->brc", nb(bf(X)), nb(dxt)), rtol=1e-12, atol=1e-12)
