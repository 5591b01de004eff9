"""Tolerance metrics shared by the parity tests.

err_max: normwise-infinity relative error max|g - r| / max(max|r|, 1e-12)
(elementwise relative error is meaningless near zero).  err_fro: Frobenius
relative error ||g - r|| / max(||r||, 1e-12), the page's backward metric.
Bounds: 2e-2 for bf16 outputs, 5e-2 for the FP8 GEMM.
"""
import numpy as np
import torch

TOL_BF16 = 2e-2
TOL_FP8 = 5e-2


def to_f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def err_max(got, ref) -> float:
    g, r = to_f64(got), to_f64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU result"
    return float(np.max(np.abs(g - r)) / max(float(np.max(np.abs(r))), 1e-12))


def err_fro(got, ref) -> float:
    g, r = to_f64(got), to_f64(ref)
    return float(np.linalg.norm((g - r).ravel()) / max(float(np.linalg.norm(r.ravel())), 1e-12))


def assert_close(got, ref, tol, what=""):
    e = err_max(got, ref)
    assert e <= tol, f"{what}: max-relative error {e:.3e} > {tol:.1e}"
    return e
