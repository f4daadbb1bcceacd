"""Shared helpers for the parity tests: error metrics and model construction."""
from __future__ import annotations

import numpy as np

# Tolerances: float32 path, max over elements of |g - o| / max(|o|, rms(o)) <= 1e-4;
# bf16 path, max |g - o| / rms(o) <= 2e-2 (rms over the compared output).
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def rms(o: np.ndarray) -> float:
    return float(np.sqrt(np.mean(np.square(o))))


def rel_err_f32(g: np.ndarray, o: np.ndarray) -> float:
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    floor = max(rms(o), 1e-30)
    return float(np.max(np.abs(g - o) / np.maximum(np.abs(o), floor)))


def rel_err_bf16(g: np.ndarray, o: np.ndarray) -> float:
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    return float(np.max(np.abs(g - o)) / max(rms(o), 1e-30))


def check(g, o, dtype: str, what: str, tol: float | None = None) -> float:
    if dtype == "f32":
        err = rel_err_f32(g, o)
        tol = TOL_F32 if tol is None else tol
    else:
        err = rel_err_bf16(g, o)
        tol = TOL_BF16 if tol is None else tol
    assert np.all(np.isfinite(np.asarray(g, dtype=np.float64))), f"{what}: non-finite GPU values"
    print(f"[parity] {what}: {err:.3e} (tol {tol:.1e})")
    assert err <= tol, f"{what}: error {err:.3e} > {tol:.1e}"
    return err
