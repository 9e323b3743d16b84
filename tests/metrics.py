"""Parity metrics and the tolerance contract shared by the tests.

Tolerances (fixed before any kernel was written, the precision-contract rule
of stratat pull #1296, "The parity discipline"):

* fp32 inputs: max-abs error <= 1e-4 on o and hT.
* bf16 inputs (the oracle sees the same bf16 values): max-abs <= 1e-2 and
  relative Frobenius error <= 2e-3, on o and on hT.

Any NaN or Inf in the result is a failure (NaN-aware metrics, same page).
"""
from __future__ import annotations

import numpy as np

TOL = {
    "f32": dict(max_abs=1e-4, rel_frob=None),
    "bf16": dict(max_abs=1e-2, rel_frob=2e-3),
}


def to_f64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def compare(got, ref, kind: str) -> dict:
    """Compare ``got`` against the fp64 ``ref`` under tolerance ``kind``."""
    got = to_f64(got)
    ref = to_f64(ref)
    if got.shape != ref.shape:
        raise AssertionError(f"shape {got.shape} != {ref.shape}")
    tol = TOL[kind]
    finite = bool(np.isfinite(got).all())
    if got.size == 0:
        return dict(max_abs=0.0, rel_frob=0.0, finite=True, ok=True, kind=kind)
    diff = got - ref
    max_abs = float(np.abs(diff).max()) if finite else float("inf")
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / den) if (finite and den > 0) else (
        0.0 if finite and float(np.linalg.norm(diff)) == 0 else float("inf"))
    ok = finite and max_abs <= tol["max_abs"]
    if tol["rel_frob"] is not None:
        ok = ok and (rel <= tol["rel_frob"] or den == 0.0 and max_abs == 0.0)
    return dict(max_abs=max_abs, rel_frob=rel, finite=finite, ok=bool(ok),
                kind=kind)


def assert_close(got, ref, kind: str, what: str = ""):
    r = compare(got, ref, kind)
    assert r["ok"], f"{what}: {r}"
    return r
