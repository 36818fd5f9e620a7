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


def check_routing(X, Wr, bias, k, g_logits, g_idx, g_w, toks=None):
    """Logits within the FP32 bound; selections valid everywhere and equal
    to the oracle's wherever the oracle's decision is certified unique.
    Returns the tokens whose routing equals the oracle's exactly."""
    o_logits, o_idx, o_w = oracle.route(X, Wr, bias, k, toks=toks)
    T = X.shape[0]
    toks = np.arange(T) if toks is None else np.asarray(toks)
    x = bits_to_f64(X[toks])
    beta = 1e-5 * (1.0 + np.abs(x) @ np.abs(Wr.astype(np.float64)))       # [n, E]
    ol, gl = o_logits[toks].astype(np.float64), g_logits[toks].astype(np.float64)
    assert np.all(np.abs(gl - ol) <= beta), np.max(np.abs(gl - ol) / beta)
    exact = []
    for n, t in enumerate(toks):
        b2 = 2 * beta[n].max()
        sel = g_idx[t]
        assert len(set(sel.tolist())) == k
        rest = np.setdiff1d(np.arange(Wr.shape[1]), sel)
        if len(rest):
            assert ol[n][sel].min() >= ol[n][rest].max() - b2
        assert np.all(np.diff(ol[n][sel]) <= b2)
        order = np.lexsort((np.arange(Wr.shape[1]), -ol[n]))
        srt = ol[n][order]
        gaps = -np.diff(srt[:min(k + 1, len(srt))])
        if np.all(gaps > b2):
            assert np.array_equal(sel, o_idx[t]), t
        if np.array_equal(sel, o_idx[t]):
            exact.append(t)
            wb = 4 * b2 * g_w[t] + 2e-6
            assert np.all(np.abs(g_w[t] - o_w[t]) <= wb)
    return np.array(exact)
