"""The tensor-core grouped GEMM (moe_grouped_gemm): dequantization inside
the GEMM is bit-exact (identity activations pull the BF16 weights through
the MMA unchanged: one exact product per output), the products match a
float64 matmul of the oracle's dequantized weights, ragged token and
feature tiles are handled, and inconsistent offsets are rejected on the
device without any out-of-range access."""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_adapter_gb300 import build, pmoe
from precision_moe_adapter_gb300 import inputs as gi
from helpers import assert_close, bits_to_f64, t2np_bits

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


def run(fmt, q, s, E, N, K, trans, A, counts):
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offsets[-1])
    out = torch.zeros((max(rows, 1), K if trans else N), dtype=torch.int16, device="cuda")
    ws = torch.zeros(pmoe.moe_grouped_gemm_ws_bytes(E, rows), dtype=torch.uint8, device="cuda")
    pmoe.moe_grouped_gemm(fmt, dev(q), dev(s), E, N, K, trans, dev(A), dev(offsets), rows, out, ws)
    st = pmoe.moe_query_status(ws)
    return t2np_bits(out)[:rows], st


def _scales_exhaustive(fmt, E, N, K):
    """Every scale whose products stay finite (an infinite weight would turn
    the zero terms of the identity contraction into NaN)."""
    ng = E * N * (K // 32)
    if fmt == gi.INT4:
        bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        f = (bits.astype(np.uint32) << 16).view(np.float32)
        with np.errstate(over="ignore", invalid="ignore"):
            fin = bits[np.isfinite(f) & (np.abs(f.astype(np.float64)) * 8 < 3.38e38)]
        return np.resize(fin, ng).reshape(E, N, K // 32)
    return np.resize(np.arange(253, dtype=np.uint8), ng).reshape(E, N, K // 32)


@pytest.mark.parametrize("fmt", [gi.INT4, gi.MXFP4, gi.FP8])
@pytest.mark.parametrize("trans", [0, 1])
def test_dequant_through_the_mma_is_bit_exact(fmt, trans):
    E, N, K = (32, 256, 256) if fmt == gi.INT4 else (8, 256, 256)
    rng = np.random.default_rng(fmt * 10 + trans)
    if fmt == gi.FP8:
        q = rng.integers(0, 256, (E, N, K), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x3C                      # no NaN codes
        q[:, 0, :] = np.tile(np.setdiff1d(np.arange(256), [0x7F, 0xFF]), 2)[:K].astype(np.uint8)
        s = (rng.random((E, N // 128, K // 128)) * 0.015 + 0.005).astype(np.float32)
    else:
        q = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
        s = _scales_exhaustive(fmt, E, N, K)
    rows_per = K if not trans else N
    eye = gi.f32_to_bf16_bits(np.eye(rows_per, dtype=np.float32))
    A = np.tile(eye, (E, 1))
    got, st = run(fmt, q, s, E, N, K, trans, A, [rows_per] * E)
    assert st == pmoe.PMOE_OK
    n_sub = n_sub_exact = 0
    # -0 weights come out of the contraction as +0 (adding +0 terms): the
    # comparison identifies the two zeros
    z = lambda x: np.where((x & 0x7FFF) == 0, 0, x).astype(np.uint16)
    for e in range(E):
        W = oracle.dequant(fmt, q[e], s[e], N, K)          # [N, K] BF16 bits
        want = z(W if trans else W.T)
        blk = z(got[e * rows_per:(e + 1) * rows_per])
        sub = ((want & 0x7F80) == 0) & ((want & 0x7F) != 0)   # BF16 subnormal weights
        assert np.array_equal(blk[~sub], want[~sub]), e
        # the MMA may flush subnormal inputs to zero; otherwise exact
        ok = (blk[sub] == want[sub]) | ((blk[sub] & 0x7FFF) == 0)
        assert ok.all(), e
        n_sub += int(sub.sum())
        n_sub_exact += int((blk[sub] == want[sub]).sum())
    print(f"subnormal weights: {n_sub}, passed through exactly: {n_sub_exact}")


@pytest.mark.parametrize("fmt", [gi.INT4, gi.MXFP4, gi.FP8])
@pytest.mark.parametrize("trans", [0, 1])
@pytest.mark.parametrize("N,K,counts", [(384, 512, [0, 1, 17, 300, 96]),
                                        (256, 256, [257, 513, 0, 16, 31]),
                                        (128, 1024, [5, 0, 0, 2])])
def test_grouped_gemm_matches_float64(fmt, trans, N, K, counts):
    E = len(counts)
    q, s = gi.gen_matrix(fmt, E, N, K, seed=N + K + sum(counts), qsid="w13", ssid="s13")
    rows = sum(counts)
    rng = np.random.default_rng(rows)
    A = gi.f32_to_bf16_bits(rng.standard_normal((rows, N if trans else K)).astype(np.float32))
    got, st = run(fmt, q, s, E, N, K, trans, A, counts)
    assert st == pmoe.PMOE_OK
    want = np.zeros(got.shape)
    r0 = 0
    for e, c in enumerate(counts):
        W = bits_to_f64(oracle.dequant(fmt, q[e], s[e], N, K))
        a = bits_to_f64(A[r0:r0 + c])
        want[r0:r0 + c] = a @ W if trans else a @ W.T
        r0 += c
    assert_close(bits_to_f64(got), want, f"gemm fmt={fmt} trans={trans}", rel_fro=3e-3, max_abs=1e-2)


def test_ragged_feature_tile():
    """N = 192 is not a multiple of the 128-row weight tile."""
    E, N, K = 2, 192, 128
    q, s = gi.gen_matrix(gi.INT4, E, N, K, seed=9, qsid="w2", ssid="s2")
    A = gi.f32_to_bf16_bits(np.random.default_rng(1).standard_normal((40, K)).astype(np.float32))
    got, st = run(gi.INT4, q, s, E, N, K, 0, A, [23, 17])
    assert st == pmoe.PMOE_OK
    want = np.concatenate([bits_to_f64(A[:23]) @ bits_to_f64(oracle.dequant(0, q[0], s[0], N, K)).T,
                           bits_to_f64(A[23:]) @ bits_to_f64(oracle.dequant(0, q[1], s[1], N, K)).T])
    assert_close(bits_to_f64(got), want, "ragged", rel_fro=3e-3, max_abs=1e-2)


@pytest.mark.parametrize("fmt", [gi.INT4, gi.MXFP4])
def test_transposed_ragged_feature_tile_is_exact(fmt):
    """Contraction over the stored rows with 320 stored columns: the last
    feature tile is 64 wide, and rows of 10 scale groups start at scale
    words that are not 4-byte aligned (MXFP4) or 8-byte aligned (INT4)."""
    E, N, K = 3, 192, 320
    q, s = gi.gen_matrix(fmt, E, N, K, seed=11, qsid="w13", ssid="s13")
    A = np.tile(gi.f32_to_bf16_bits(np.eye(N, dtype=np.float32)), (E, 1))
    got, st = run(fmt, q, s, E, N, K, 1, A, [N] * E)
    assert st == pmoe.PMOE_OK
    z = lambda x: np.where((x & 0x7FFF) == 0, 0, x).astype(np.uint16)
    for e in range(E):
        want = z(oracle.dequant(fmt, q[e], s[e], N, K))
        assert np.array_equal(z(got[e * N:(e + 1) * N]), want), e


@pytest.mark.parametrize("offsets", [[0, 5, 3, 8], [0, 4, 8, 9], [1, 4, 6, 8]])
def test_inconsistent_offsets_are_rejected(offsets):
    E, N, K, rows = 3, 128, 128, 8
    q, s = gi.gen_matrix(gi.INT4, E, N, K, seed=2, qsid="w2", ssid="s2")
    A = torch.zeros((rows, K), dtype=torch.int16, device="cuda")
    out = torch.full((rows, N), 7, dtype=torch.int16, device="cuda")
    ws = torch.zeros(pmoe.moe_grouped_gemm_ws_bytes(E, rows), dtype=torch.uint8, device="cuda")
    pmoe.moe_grouped_gemm(gi.INT4, dev(q), dev(s), E, N, K, 0, A,
                          dev(np.array(offsets, np.int32)), rows, out, ws)
    assert pmoe.moe_query_status(ws) == pmoe.PMOE_ERR_BAD_INDEX
    assert torch.all(out == 7)
