"""Attention tolerance: max abs error 2e-3 and max rel error 1e-2 against fp64.

Reading used, each part asserted on its own:
  * absolute: |out - ref| <= 2e-3 on every element whose 16-bit output format can
    represent the bound, i.e. where half an ulp of fp16 / bf16 at |ref| is at most
    1e-3 (rounding to bf16 alone exceeds 2e-3 once |ref| >= 0.5);
  * relative: |out - ref| / |ref| <= 1e-2 on every element with |ref| >= 0.1 (a
    relative error means nothing at ref ~ 0).
Every element falls under at least one of the two: an element exempt from the
absolute bound has |ref| >= 0.5 (fp16: >= 4) and so is held to the relative one.
"""
import numpy as np

ATOL = 2e-3
RTOL = 1e-2
REL_FLOOR = 0.1
MANT = {"fp16": 10, "bf16": 7}


def half_ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    mant = MANT[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -24)))
    return 2.0 ** (e - mant - 1)


def check(out: np.ndarray, ref: np.ndarray, dtype: str, what: str = "") -> dict:
    """Assert both bounds; return the observed maxima (abs over the elements the
    absolute bound covers and over all, rel over |ref| >= 0.1)."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert out.shape == ref.shape, (out.shape, ref.shape)
    assert np.isfinite(ref).all(), f"{what}: non-finite oracle output"
    assert np.isfinite(out).all(), f"{what}: non-finite output ({np.isnan(out).sum()} NaN)"
    err = np.abs(out - ref)
    strict = half_ulp(ref, dtype) <= 1e-3
    big = np.abs(ref) >= REL_FLOOR
    assert (strict | big).all(), f"{what}: an element is under neither bound"
    max_abs = float(err[strict].max()) if strict.any() else 0.0
    assert max_abs <= ATOL, (
        f"{what}: max abs error {max_abs:.3e} > {ATOL} (at ref "
        f"{ref[strict][np.argmax(err[strict])]:.4f})")
    rel = err[big] / np.abs(ref[big])
    max_rel = float(rel.max()) if big.any() else 0.0
    assert max_rel <= RTOL, (
        f"{what}: max rel error {max_rel:.3e} > {RTOL} over |ref| >= {REL_FLOOR} (at ref "
        f"{ref[big][np.argmax(rel)]:.4f})")
    return {"max_abs": max_abs, "max_abs_all": float(err.max()) if err.size else 0.0,
            "max_rel_big": max_rel, "n": int(err.size)}
