"""Pins of the oracle's element formats and BF16 rounding against facts
other than the oracle: brute-force nearest-BF16 search, torch's library
conversions, and format tables from the published specs (tests/golden)."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _all_finite_bf16():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    keep = np.isfinite(f)
    return bits[keep], f[keep].astype(np.float64)


def _nearest_bf16_bruteforce(v):
    """Nearest BF16 to each double by search over every finite BF16 value,
    ties to the even bit pattern, overflow to inf past the rounding edge."""
    bits, vals = _all_finite_bf16()
    pos = vals >= 0
    pb, pv = bits[pos & ~np.signbit(vals)], vals[pos & ~np.signbit(vals)]
    order = np.argsort(pv, kind="stable")
    pb, pv = pb[order], pv[order]
    out = np.empty(v.shape, np.uint16)
    maxv = pv[-1]
    edge = maxv + (maxv - pv[-2]) / 2          # halfway to 2^128
    for i, x in enumerate(v):
        a = abs(x)
        sign = 0x8000 if np.signbit(x) else 0
        if a >= edge:
            out[i] = sign | 0x7F80
            continue
        j = np.searchsorted(pv, a)
        cands = [c for c in (j - 1, j) if 0 <= c < len(pv)]
        best = min(cands, key=lambda c: (abs(pv[c] - a), int(pb[c]) & 1))
        out[i] = sign | int(pb[best])
    return out


def test_bf16_round_bruteforce():
    rng = np.random.default_rng(1)
    _, vals = _all_finite_bf16()
    vals = vals[vals > 0]
    vals.sort()
    mids = (vals[:-1] + vals[1:]) / 2                         # exact ties
    pick = rng.choice(len(mids), 400, replace=False)
    v = np.concatenate([
        mids[pick], -mids[pick[:50]],
        rng.standard_normal(400) * 10.0 ** rng.integers(-45, 39, 400),
        np.nextafter(mids[pick[:100]], np.inf), np.nextafter(mids[pick[:100]], -np.inf),
        [0.0, -0.0, 2.0 ** -133, 2.0 ** -134, 2.0 ** -134 * 1.0000001, 3.4e38, 3.39e38, 1e39,
         2.0 ** 128 * (1 - 2.0 ** -9), 2.0 ** 128 * (1 - 2.0 ** -8)],
    ])
    got = oracle.bf16_round(v)
    want = _nearest_bf16_bruteforce(v)
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:10]


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(2)
    f = (rng.standard_normal(5000) * 10.0 ** rng.integers(-40, 38, 5000)).astype(np.float32)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_round(f.astype(np.float64)), want)


def test_int4_dequant_exhaustive():
    """All 16 nibbles x all 65280 finite BF16 scales, against
    torch(fp32(q) * fp32(s)).to(bf16) -- the product is exact in FP32."""
    sbits, _ = _all_finite_bf16()
    N, K = len(sbits), 32
    q_vals = np.tile(np.arange(16, dtype=np.uint8), 2)              # 32 elements / row
    lo, hi = q_vals[0::2], q_vals[1::2]
    q = np.tile((lo | (hi << 4)).astype(np.uint8), (N, 1))           # [N, 16] bytes
    s = sbits.reshape(N, 1)
    got = oracle.dequant(oracle.INT4, q, s, N, K)
    signed = np.where(q_vals >= 8, q_vals.astype(np.int32) - 16, q_vals.astype(np.int32))
    sf = torch.from_numpy((sbits.astype(np.uint32) << 16).view(np.float32).copy())
    prod = torch.from_numpy(signed.astype(np.float32))[None, :] * sf[:, None]
    want = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def _load_e2m1():
    vals = {}
    with open(os.path.join(GOLD, "e2m1_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            vals[int(c)] = float(v)
    return vals


def test_mxfp4_dequant_exhaustive():
    """All 16 E2M1 codes x all 255 finite E8M0 scales, against the spec's
    value table times 2^(u-127), rounded by torch (exact unless out of the
    BF16 range)."""
    tab = _load_e2m1()
    codes = np.arange(16)
    mag = np.array([tab[c & 7] for c in codes])
    val = np.where(codes >= 8, -mag, mag)
    val = np.where(codes == 8, -0.0, val)
    N, K = 255, 32
    q_vals = np.tile(np.arange(16, dtype=np.uint8), 2)
    q = np.tile((q_vals[0::2] | (q_vals[1::2] << 4)).astype(np.uint8), (N, 1))
    s = np.arange(255, dtype=np.uint8).reshape(N, 1)
    got = oracle.dequant(oracle.MXFP4, q, s, N, K)
    want = np.empty((N, K), np.uint16)
    for u in range(255):
        row = np.array([np.ldexp(val[c], u - 127) for c in np.tile(codes, 2)])
        with np.errstate(over="ignore"):
            want[u] = torch.from_numpy(row).to(torch.float32).to(torch.bfloat16) \
                .view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    # E8M0 255 is NaN
    nan = oracle.dequant(oracle.MXFP4, q[:1], np.array([[255]], np.uint8), 1, K)
    assert np.all((nan & 0x7F80) == 0x7F80) and np.all((nan & 0x7F) != 0)


def test_e4m3_decode_matches_torch_and_spec():
    got = oracle.e4m3_values()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))
    with open(os.path.join(GOLD, "e4m3_special.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            c, v = int(c, 16), float(v)
            if np.isnan(v):
                assert np.isnan(got[c])
            else:
                assert got[c] == v and np.signbit(got[c]) == np.signbit(v)


def test_fp8_dequant_double_rounding():
    """All 256 codes x 10^4 seeded FP32 scales: W = bf16(fp32(v * s)),
    against torch's FP32 multiply then BF16 conversion."""
    rng = np.random.default_rng(3)
    ns = 10000
    scales = (rng.random(ns) * 0.015 + 0.005).astype(np.float32)
    scales[:100] = (rng.standard_normal(100) * 10.0 ** rng.integers(-30, 30, 100)).astype(np.float32)
    # one [128, 128] block per scale: rows 128*i..128*i+127, K = 256 (2 blocks)
    codes = np.arange(256, dtype=np.uint8)
    nblk = 40
    for base in range(0, ns, nblk):
        sc = scales[base:base + nblk]
        N, K = 128 * len(sc), 256
        q = np.tile(codes, (N, 1))
        s = np.stack([sc, sc], axis=1).reshape(len(sc), 2)
        got = oracle.dequant(oracle.FP8, q, s, N, K)
        v = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32)
        prod = v[None, None, :] * torch.from_numpy(sc)[:, None, None]
        want = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        want = np.broadcast_to(want[:, :, :], (len(sc), 1, 256)).reshape(len(sc), 256)
        got_rows = got.reshape(len(sc), 128, 256)
        nanmask = np.isnan(v.numpy())
        for i in range(len(sc)):
            g = got_rows[i]
            assert np.all(g == g[0])                       # rows of a block agree
            assert np.array_equal(g[0][~nanmask], want[i][~nanmask])
            assert np.all((g[0][nanmask] & 0x7F80) == 0x7F80)


def _nibbles(q):
    lo, hi = (q & 15).astype(np.int32), (q >> 4).astype(np.int32)
    n = np.stack([lo, hi], axis=-1).reshape(q.shape[0], -1)
    return n


def test_multi_group_scale_indexing():
    """Several scale groups / blocks per row with distinct scales: each
    element must use the scale of its own group (torch reference)."""
    rng = np.random.default_rng(4)
    N, K = 8, 256
    q = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    n = _nibbles(q)
    # INT4
    s = gi_bf16(rng.random((N, K // 32)) * 0.015 + 0.005)
    sf = torch.from_numpy((s.astype(np.uint32) << 16).view(np.float32))
    qi = torch.from_numpy(np.where(n >= 8, n - 16, n).astype(np.float32))
    want = (qi * sf.repeat_interleave(32, dim=1)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.dequant(oracle.INT4, q, s, N, K), want)
    # MXFP4
    tab = _load_e2m1()
    e = rng.integers(119, 124, (N, K // 32)).astype(np.uint8)
    mag = np.vectorize(lambda c: tab[c & 7])(n)
    val = np.where(n >= 8, -mag, mag) * np.ldexp(1.0, np.repeat(e.astype(np.int32) - 127, 32, axis=1))
    want = torch.from_numpy(val).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.dequant(oracle.MXFP4, q, e, N, K), want)
    # FP8, [128,128] blocks
    N8, K8 = 256, 384
    c8 = rng.integers(0, 256, (N8, K8), dtype=np.uint8)
    c8[c8 == 0x7F] = 0x10
    c8[c8 == 0xFF] = 0x90
    s8 = (rng.random((2, 3)) * 0.015 + 0.005).astype(np.float32)
    v = torch.from_numpy(c8).view(torch.float8_e4m3fn).to(torch.float32)
    sb = torch.from_numpy(s8).repeat_interleave(128, 0).repeat_interleave(128, 1)
    want = (v * sb).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.dequant(oracle.FP8, c8, s8, N8, K8), want)


def gi_bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
