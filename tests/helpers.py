"""Shared helpers of the test suite (conversions and the tolerance of the
layer's floating-point outputs)."""
import numpy as np

import oracle

# Tolerance for BF16 outputs and gradients: relative Frobenius error and a
# per-element bound relative to the reference magnitude.
REL_FRO = 5e-3
MAX_ABS = 2e-2


def bits_to_f64(h) -> np.ndarray:
    h = np.ascontiguousarray(h).view(np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def t2np_bits(t) -> np.ndarray:
    """int16 torch tensor holding BF16 bits -> numpy uint16."""
    return t.detach().cpu().numpy().view(np.uint16)


def assert_close(got, ref, what="", rel_fro=REL_FRO, max_abs=MAX_ABS):
    """Relative Frobenius error <= rel_fro, and every element within
    max_abs * (1 + |ref|): the tolerance stated for the layer's BF16
    outputs and gradients."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    den = np.linalg.norm(ref)
    err = np.linalg.norm(got - ref)
    rel = err / den if den > 0 else err
    bound = max_abs * (1.0 + np.abs(ref))
    bad = np.abs(got - ref) > bound
    assert rel <= rel_fro, f"{what}: relative Frobenius error {rel:.3e} > {rel_fro}"
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond {max_abs}(1+|ref|), "
                           f"worst {np.max(np.abs(got - ref) - bound):.3e}")
    return rel


def check_cayley(Rb_bits, Rf, R64, b):
    """Device Cayley map against the FP64 one: R_f32 within 4 b 2^-24 (FP32
    elimination on b x b blocks of norm about 1), and R_bf16 = bf16(R_f32):
    rounding is monotone, so it lies between the roundings of R - eps and
    R + eps, and equals bf16 of the exact R wherever those two agree.
    Returns the number of elements where they do not (where the FP32 error
    bound alone cannot fix the BF16 value)."""
    eps = 4 * b * 2.0 ** -24
    rf = np.asarray(Rf, np.float64)
    assert np.max(np.abs(rf - R64)) < eps
    rb = bits_to_f64(Rb_bits)
    lo = bits_to_f64(oracle.bf16_round((R64 - eps).ravel())).reshape(R64.shape)
    hi = bits_to_f64(oracle.bf16_round((R64 + eps).ravel())).reshape(R64.shape)
    assert np.all((rb >= lo) & (rb <= hi))
    ref = bits_to_f64(oracle.bf16_round(R64.ravel())).reshape(R64.shape)
    assert np.all((rb == ref) | (lo != hi))
    return int(np.sum(lo != hi))


def check_topk(g_logits, g_idx, g_w, k, toks=None):
    """The device's selection and weights against the oracle's top-k and
    softmax applied to the device's own logits (bias included): idx bit for
    bit, w within 1e-6 relative."""
    o_idx, o_w = oracle.topk(g_logits, k, toks=toks)
    rows = slice(None) if toks is None else np.asarray(toks)
    assert np.array_equal(g_idx[rows], o_idx[rows])
    assert np.all(np.abs(g_w[rows].astype(np.float64) - o_w[rows]) <= 1e-6 * np.abs(o_w[rows]))


def check_routing(X, Wr, bias, k, g_logits, g_idx, g_w, toks=None):
    """Device routing from the fast router mode:
      - logits within the FP32 bound 1e-5 (1 + sum |x w|) of the oracle's
        FP64 logits;
      - idx bit-exact and w within 1e-6 relative against the oracle's top-k
        and softmax applied to the device's own logits;
      - against the oracle's own routing, a token may differ only where the
        oracle's order near the k-th place is not certified (two logits
        within twice the bound).
    Returns the tokens whose routing equals the oracle's own exactly."""
    o_logits, o_idx, o_w = oracle.route(X, Wr, bias, k, toks=toks)
    T = X.shape[0]
    toks = np.arange(T) if toks is None else np.asarray(toks)
    check_topk(g_logits, g_idx, g_w, k, toks=toks)
    x = bits_to_f64(X[toks])
    beta = 1e-5 * (1.0 + np.abs(x) @ np.abs(Wr.astype(np.float64)))       # [n, E]
    ol, gl = o_logits[toks].astype(np.float64), g_logits[toks].astype(np.float64)
    assert np.all(np.abs(gl - ol) <= beta), np.max(np.abs(gl - ol) / beta)
    exact = []
    for n, t in enumerate(toks):
        if np.array_equal(g_idx[t], o_idx[t]):
            exact.append(t)
            continue
        # a flip: the oracle's own order must have a near-tie within the
        # first k + 1 places
        b2 = 2 * beta[n].max()
        order = np.lexsort((np.arange(Wr.shape[1]), -ol[n]))
        gaps = -np.diff(ol[n][order][:min(k + 1, len(order))])
        assert np.any(gaps <= b2), (t, gaps.min(), b2)
    return np.array(exact)

