"""Dense bypass-base-weight-grad linear with the OFT adapter, through the
C ABI, against the oracle: INT4 / MXFP4 / FP8 weights, with and without the
adapter, ragged row counts."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bits_to_f64, t2np_bits
from precision_moe_adapter_gb300 import build, pmoe
from precision_moe_adapter_gb300 import inputs as gi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    pmoe.lib()
    oracle.build()


def dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if t.dtype == torch.uint16:
        t = t.view(torch.int16)
    return t.cuda()


@pytest.mark.parametrize("fmt,rows,N,K,b,adapter", [
    (gi.INT4, 300, 384, 512, 64, True),
    (gi.INT4, 37, 256, 192, 32, True),
    (gi.INT4, 129, 128, 256, 32, False),
    (gi.MXFP4, 200, 256, 384, 64, True),
    (gi.FP8, 96, 256, 256, 128, True),
    (gi.INT4, 1, 256, 256, 16, True),
])
def test_dense_linear_matches_the_oracle(fmt, rows, N, K, b, adapter):
    q, s = gi.gen_matrix(fmt, 1, N, K, seed=rows + N, qsid="w2", ssid="s2")
    q, s = q[0], s[0]
    rng = np.random.default_rng(rows)
    X = gi.f32_to_bf16_bits(rng.standard_normal((rows, K)).astype(np.float32))
    dY = gi.f32_to_bf16_bits(0.1 * rng.standard_normal((rows, N)).astype(np.float32))
    R = None
    if adapter:
        S = gi.gen_skew(1, K, b, rows, "S_up", 0.01)[0]
        R = gi.f32_to_bf16_bits(oracle.cayley(S).astype(np.float32))
    ws = torch.zeros(pmoe.dense_linear_ws_bytes(rows, N, K), dtype=torch.uint8, device="cuda")
    Y = torch.empty((rows, N), dtype=torch.int16, device="cuda")
    dX = torch.empty((rows, K), dtype=torch.int16, device="cuda")
    dR = torch.empty((K // b, b, b), dtype=torch.float32, device="cuda") if adapter else None
    qd, sd, Rd, Xd = dev(q), dev(s), None if R is None else dev(R), dev(X)
    pmoe.dense_linear_forward(fmt, qd, sd, N, K, b, Rd, rows, Xd, Y, ws)
    pmoe.dense_linear_backward(fmt, qd, sd, N, K, b, Rd, rows, Xd, dev(dY), dX, dR, ws)
    assert pmoe.moe_query_status(ws) == pmoe.PMOE_OK
    _, Y64 = oracle.dense_forward(fmt, q, s, N, K, b, R, X)
    ob = oracle.dense_backward(fmt, q, s, N, K, b, R, X, dY)
    assert_close(bits_to_f64(t2np_bits(Y)), Y64, "dense Y")
    assert_close(bits_to_f64(t2np_bits(dX)), ob["dX64"], "dense dX")
    if adapter:
        assert_close(dR.cpu().numpy().astype(np.float64), ob["dR"], "dense dR")


def test_dense_linear_zero_adapter_is_the_base():
    """R = I (from S = 0) gives exactly the adapter-less projection."""
    fmt, rows, N, K, b = gi.INT4, 64, 256, 256, 64
    q, s = gi.gen_matrix(fmt, 1, N, K, seed=4, qsid="w2", ssid="s2")
    X = gi.f32_to_bf16_bits(np.random.default_rng(4).standard_normal((rows, K)).astype(np.float32))
    I = gi.f32_to_bf16_bits(oracle.cayley(np.zeros((K // b, b, b))).astype(np.float32))
    ws = torch.zeros(pmoe.dense_linear_ws_bytes(rows, N, K), dtype=torch.uint8, device="cuda")
    Y0 = torch.empty((rows, N), dtype=torch.int16, device="cuda")
    Y1 = torch.empty_like(Y0)
    pmoe.dense_linear_forward(fmt, dev(q[0]), dev(s[0]), N, K, b, None, rows, dev(X), Y0, ws)
    pmoe.dense_linear_forward(fmt, dev(q[0]), dev(s[0]), N, K, b, dev(I), rows, dev(X), Y1, ws)
    assert torch.equal(Y0, Y1)
