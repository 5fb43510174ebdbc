"""Comparison helpers for the parity tests (CUDA path vs the CPU oracle).

Tolerances: elementwise |gpu - ref| <= rtol*|ref| + atol.
  * forward, fp32 features: rtol 1e-5. atol 1e-6 covers outputs that cancel
    to near 0 (signed DCNv4-style weights).
  * backward (atomically accumulated): rtol 1e-4, atol 1e-6.
  * bf16 features: rtol 2e-2. The oracle reads the same bf16 values exactly
    widened, so the real error is far smaller; the test also reports it.
"""
from __future__ import annotations

import numpy as np
import torch

EPS32 = float(np.finfo(np.float32).eps)

TOL = {
    "f32": {"out": (1e-5, 1e-6), "grad_feat": (1e-4, 1e-6), "grad_loc": (1e-4, 1e-6),
            "grad_weight": (1e-4, 1e-6)},
    "bf16": {"out": (2e-2, 1e-6), "grad_feat": (2e-2, 1e-6), "grad_loc": (2e-2, 1e-6),
             "grad_weight": (2e-2, 1e-6)},
}


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def violations(gpu: np.ndarray, ref: np.ndarray, rtol: float, atol, name: str = ""):
    """Return (count, message) for elements outside |g-r| <= rtol*|r| + atol."""
    g = np.asarray(gpu, np.float64).ravel()
    r = np.asarray(ref, np.float64).ravel()
    assert g.shape == r.shape, (name, g.shape, r.shape)
    a = np.asarray(atol, np.float64).ravel() if np.ndim(atol) else atol
    err = np.abs(g - r)
    lim = rtol * np.abs(r) + a
    bad = ~(err <= lim)  # NaN counts as a violation
    n = int(bad.sum())
    if n == 0:
        return 0, ""
    i = int(np.argmax(np.where(bad, err - lim, -np.inf)))
    return n, (f"{name}: {n}/{g.size} outside tolerance (rtol={rtol}); worst at {i}: "
               f"gpu={g[i]!r} ref={r[i]!r} |err|={err[i]:.3e} limit={np.ravel(lim)[i]:.3e}")


def max_rel(gpu: np.ndarray, ref: np.ndarray, floor: float = 1e-3) -> float:
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), floor))) if g.size else 0.0


def assert_close(gpu, ref, kind: str, name: str, atol_extra=None):
    rtol, atol = TOL[kind][name]
    if atol_extra is not None:
        atol = atol + atol_extra
    n, msg = violations(gpu, ref, rtol, atol, name)
    assert n == 0, msg
