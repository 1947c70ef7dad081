"""Attention tolerance: max abs error 2e-3 and max rel error 1e-2 against fp64.

Reading used (both parts are asserted):
  * every element: |out - ref| <= 2e-3 + 1e-2 * |ref|   (abs and rel bounds combined
    elementwise, the usual atol/rtol form; a bare relative bound is meaningless at
    ref ~ 0 and a bare 2e-3 absolute bound cannot hold once half an ulp of the
    16-bit output format exceeds it, e.g. bf16 at |ref| >= 0.5);
  * strict absolute bound |out - ref| <= 2e-3 on every element whose output
    format can represent it, i.e. where half an ulp of fp16 / bf16 at |ref| is at
    most 1e-3.
"""
import numpy as np

ATOL = 2e-3
RTOL = 1e-2
MANT = {"fp16": 10, "bf16": 7}


def half_ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    mant = MANT[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -24)))
    return 2.0 ** (e - mant - 1)


def check(out: np.ndarray, ref: np.ndarray, dtype: str, what: str = "") -> dict:
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert out.shape == ref.shape, (out.shape, ref.shape)
    assert np.isfinite(ref).all(), f"{what}: non-finite oracle output"
    assert np.isfinite(out).all(), f"{what}: non-finite output ({np.isnan(out).sum()} NaN)"
    err = np.abs(out - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} elements beyond 2e-3 + 1e-2|ref|; worst "
                           f"err {err[bad].max():.3e} at ref {ref[bad][np.argmax(err[bad])]:.4f}")
    strict = half_ulp(ref, dtype) <= 1e-3
    if strict.any():
        assert err[strict].max() <= ATOL, f"{what}: strict abs {err[strict].max():.3e} > 2e-3"
    big = np.abs(ref) >= 0.1
    return {
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_rel_big": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
        "n": int(err.size),
    }
