"""Shared helpers of the test suite (conversions and the tolerance of the
layer's floating-point outputs)."""
import numpy as np

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
