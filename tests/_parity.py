"""Element-wise comparison of CUDA results with the fp64 oracle.

Tolerances (per element, o = oracle value, g = GPU value):
  fp32 storage:  |g - o| <= 1e-5 * |o| + 1e-6
  bf16 storage:  |g - o| <= 1e-2 + 2e-2 * |o|
The fp32 bound is a relative error of 1e-5 with a 1e-6 floor where
cancellation makes |o| tiny; the bf16 bound is a relative error of 2e-2 with
an absolute floor of 1e-2.  Both apply to every output (y, dx, dw, dz, dU, db).
"""
import numpy as np
import torch


def tol(dtype: str):
    return (1e-5, 1e-6) if dtype == "f32" else (2e-2, 1e-2)


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def assert_close(got, ref, dtype: str, what: str = ""):
    g = to_np(got).reshape(np.shape(ref))
    r = np.asarray(ref, dtype=np.float64)
    rel, ab = tol(dtype)
    err = np.abs(g - r)
    lim = rel * np.abs(r) + ab
    bad = ~(err <= lim)  # also catches NaN
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first at {i}: "
            f"gpu={g[i]!r} oracle={r[i]!r}; max abs err {np.nanmax(err):.3e}; "
            f"normwise {np.nanmax(err) / max(np.abs(r).max(), 1e-300):.3e}")
    return float(err.max()) if err.size else 0.0
