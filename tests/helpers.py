"""Shared helpers for the parity tests: the error metrics."""
from __future__ import annotations

import numpy as np

# Tolerances (written here, used by every parity test):
#   float32 path: max over elements of |g - o| / max(|o|, rms(o)) <= 1e-4;
#   bf16 path:    max over elements of |g - o| / rms(o) <= 2e-2, rms over the compared output.
# A result the library STORES in bf16 carries its own rounding: a value computed
# exactly and then correctly rounded to bf16 is off by up to half an ulp, which
# for |o| >= 8 is already 2^-5 ~ 2.8e-2 * rms for unit-rms outputs.  For such
# outputs the bar applies to the computation: the half-ulp of bf16 at the value
# is allowed on top, |g - o| <= 2e-2 rms(o) + ulp_bf16(|o|) / 2.  Results stored
# in float32 (the pooled output, the MoE PFFN output) are held to the bare bound.
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def rms(o: np.ndarray) -> float:
    return float(np.sqrt(np.mean(np.square(o))))


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) at |x|."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def rel_err_f32(g: np.ndarray, o: np.ndarray) -> float:
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    floor = max(rms(o), 1e-30)
    return float(np.max(np.abs(g - o) / np.maximum(np.abs(o), floor)))


def rel_err_bf16(g: np.ndarray, o: np.ndarray, stored_bf16: bool = False, both_stored: bool = False) -> float:
    """max |g - o| / rms(o); stored_bf16: g was rounded to bf16 by the library (half an
    ulp allowed); both_stored: g and o are two such results (half an ulp each)."""
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    d = np.abs(g - o)
    if stored_bf16 or both_stored:
        # (1 + 2^-14): the store rounds a float32 value, not the exact one
        d = np.maximum(d - half_ulp_bf16(np.maximum(np.abs(o), np.abs(g))) * (1 + 2.0 ** -14) * (2 if both_stored else 1),
                       0.0)
    return float(np.max(d) / max(rms(o), 1e-30))


def _as_np(g):
    try:
        import torch
        if isinstance(g, torch.Tensor):
            return g.detach().to("cpu", torch.float64).numpy(), g.dtype == torch.bfloat16
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(g, dtype=np.float64), False


def check(g, o, dtype: str, what: str, tol: float | None = None, both_stored: bool = False) -> float:
    """g: GPU result (torch tensor or array), o: oracle result; dtype: the path ("f32" or "bf16").
    both_stored: o is itself a bf16-stored GPU result (a comparison of two paths)."""
    g, stored_bf16 = _as_np(g)
    if dtype == "f32":
        err = rel_err_f32(g, o)
        tol = TOL_F32 if tol is None else tol
    else:
        err = rel_err_bf16(g, o, stored_bf16, both_stored=both_stored and stored_bf16)
        tol = TOL_BF16 if tol is None else tol
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    raw = rel_err_bf16(g, o) if dtype != "f32" else err
    print(f"[parity] {what}: {err:.3e} (tol {tol:.1e}; max|g-o|/rms {raw:.3e}{', bf16-stored' if stored_bf16 else ''})")
    assert err <= tol, f"{what}: error {err:.3e} > {tol:.1e}"
    return err
