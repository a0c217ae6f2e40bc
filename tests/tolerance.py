"""Parity tolerances for bf16-in / fp32-accumulate results: max-abs error
2e-2 and relative L2 error 5e-3, against the fp64 oracle in its
precision-model mode (``bf16_operands=True``: every contraction input rounded
to bf16, everything else exact), so that the bound measures an
implementation's own arithmetic, not the rounding the precision model itself
implies.

Readings that make the max-abs bound meaningful for every output:
 * weight gradients (dWqkv, dWo, fp32) sum over all L tokens and grow like
   sqrt(L): the bound applies to the error divided by max(1, RMS of the
   oracle tensor);
 * a bf16-typed output of magnitude m carries its own storage rounding of up
   to m * 2^-9, which alone exceeds 2e-2 once m > 10: for bf16 outputs the
   bound applies to the error divided by max(1, |oracle element|) (identical
   to the raw bound wherever |oracle| <= 1).
The relative L2 bound applies unchanged to every output.

Against the plain fp64 definition (no rounding anywhere) an implementation
also carries the precision model's own deviation.  ``assert_close_plain``
bounds that comparison by the triangle inequality, |got - exact| <=
|got - model| + |model - exact|: each figure (scaled max-abs and rel-L2) is
at most the model's own deviation from the exact result plus the tolerance
above.  (At long sequences the bf16 rounding of Q and K alone moves the
model's late rows by several 1e-3 relative, so the stated rel-L2 cannot
hold against the exact result there by itself.)
"""

import numpy as np

MAX_ABS = 2e-2
REL_L2 = 5e-3


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    return max_abs, rel, rms


def scaled_max_abs(got, ref, weight_grad=False):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    err = np.abs(got - ref)
    if weight_grad:
        return float(np.max(err) / max(1.0, float(np.sqrt(np.mean(ref ** 2)))))
    return float(np.max(err / np.maximum(1.0, np.abs(ref))))


def report(name, got, ref, weight_grad=False, against="model"):
    """One line of figures (printed; shown by pytest -s or -rA)."""
    max_abs, rel, rms = errors(got, ref)
    scaled = scaled_max_abs(got, ref, weight_grad)
    print(f"[parity] {name} vs {against}: raw max-abs {max_abs:.3e}, scaled max-abs {scaled:.3e}, "
          f"rel-L2 {rel:.3e}, RMS(ref) {rms:.3e}")
    return max_abs, scaled, rel


def assert_close(got, ref, name, weight_grad=False):
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{name}: non-finite values"
    max_abs, scaled, rel = report(name, got, ref, weight_grad)
    assert scaled <= MAX_ABS, f"{name}: scaled max-abs {scaled:.3e} (raw {max_abs:.3e}) > {MAX_ABS}"
    assert rel <= REL_L2, f"{name}: rel-L2 {rel:.3e} > {REL_L2}"
    return max_abs, rel


def assert_close_plain(got, exact, model, name, weight_grad=False):
    """got against the plain fp64 definition `exact`, given the precision
    model's result `model` for the same inputs (see the module docstring)."""
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{name}: non-finite values"
    max_abs, scaled, rel = report(name, got, exact, weight_grad, against="plain fp64")
    inherent = scaled_max_abs(model, exact, weight_grad)
    _, rel_inherent, _ = errors(model, exact)
    print(f"[parity] {name}: the precision model itself vs plain fp64: scaled max-abs {inherent:.3e}, "
          f"rel-L2 {rel_inherent:.3e}")
    assert rel <= rel_inherent + REL_L2, (
        f"{name}: rel-L2 against the plain definition {rel:.3e} > the precision model's own "
        f"{rel_inherent:.3e} + {REL_L2}")
    assert scaled <= inherent + MAX_ABS, (
        f"{name}: scaled max-abs against the plain definition {scaled:.3e} > the precision model's own "
        f"{inherent:.3e} + {MAX_ABS}")
    return max_abs, rel


def assert_max_abs(got, ref, name, weight_grad=False):
    """Element-wise bound only (for hand-picked edge rows, which are not a
    uniform sample of the tensor and so say nothing about its rel-L2)."""
    scaled = scaled_max_abs(got, ref, weight_grad)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{name}: non-finite values"
    print(f"[parity] {name} (edge rows): scaled max-abs {scaled:.3e}")
    assert scaled <= MAX_ABS, f"{name}: scaled max-abs {scaled:.3e} > {MAX_ABS}"
    return scaled
