"""Shared helpers for the parity tests: the error metrics and the bf16 rounding check."""
from __future__ import annotations

import numpy as np

# Tolerances (written here, used by every parity test):
#   float32 path: max over elements of |g - o| / max(|o|, rms(o)) <= 1e-4;
#   bf16 path:    max over elements of |g - o| / rms(o) <= 2e-2, rms over the compared output.
# Both bars apply to the computation.  Where a bf16 context stores an output in
# bf16, the tests ask the library for the same output in float32 (out_dtype
# RM_F32: the values before their last rounding), hold that to the bar, and
# check the bf16 output bit for bit against round-to-nearest-even of it
# (assert_bf16_rounding).
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
    """max |g - o| / rms(o)."""
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    return float(np.max(np.abs(g - o)) / max(rms(o), 1e-30))


def _as_np(g):
    try:
        import torch
        if isinstance(g, torch.Tensor):
            return g.detach().to("cpu", torch.float64).numpy(), g.dtype == torch.bfloat16
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(g, dtype=np.float64), False


def check(g, o, dtype: str, what: str, tol: float | None = None) -> float:
    """g: GPU result (torch tensor or array), o: oracle result; dtype: the path ("f32" or "bf16").
    The bare bar of the path, with no allowance for the storage format."""
    g, stored_bf16 = _as_np(g)
    if dtype == "f32":
        err = rel_err_f32(g, o)
        tol = TOL_F32 if tol is None else tol
    else:
        err = rel_err_bf16(g, o)
        tol = TOL_BF16 if tol is None else tol
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    print(f"[parity] {what}: {err:.3e} (tol {tol:.1e}{', bf16-stored' if stored_bf16 else ''})")
    assert err <= tol, f"{what}: error {err:.3e} > {tol:.1e}"
    return err


def assert_bf16_rounding(g_bf16, g_f32, what: str) -> None:
    """The bf16 output equals round-to-nearest-even of the float32 output of the same
    computation, bit for bit (torch's float32 -> bfloat16 conversion rounds to nearest even)."""
    import torch
    assert g_bf16.dtype == torch.bfloat16 and g_f32.dtype == torch.float32, what
    want = g_f32.to(torch.bfloat16)
    same = torch.eq(g_bf16.view(torch.int16), want.view(torch.int16))
    n_bad = int((~same).sum().item())
    print(f"[parity] {what}: bf16 output == RNE(float32 output) for {g_bf16.numel() - n_bad}/{g_bf16.numel()}")
    assert n_bad == 0, f"{what}: {n_bad} bf16 values differ from the rounded float32 result"
