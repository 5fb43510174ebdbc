"""Comparison helpers for the parity tests (CUDA path vs the CPU oracle).

Tolerances: elementwise |gpu - ref| <= rtol*|ref| + atol.
  * forward, fp32 features: rtol 1e-5. atol 1e-6 covers outputs that cancel
    to near 0 (signed DCNv4-style weights).
  * backward (atomically accumulated): rtol 1e-4, atol 1e-6.
  * bf16 features: rtol 2e-2. The oracle reads the same bf16 values exactly
    widened, so the real error is far smaller; the test also reports it.

grad_loc and grad_weight are sums of signed products that can cancel to
almost nothing. grad_loc holds differences of corner values scaled by the
map width, over D channels, S scales and G groups. grad_weight holds signed
grad_out times the sampled values. Where they cancel, a relative bound
measures only the cancellation. For these two outputs the absolute part
therefore also gets the standard error bound of an fp32 sum:
    kappa * u * M,   with u = 2**-24 (fp32 unit roundoff),
where M is the sum of the absolute values of every product in the element,
and kappa bounds the number of sequential fp32 roundings along the kernel's
longest accumulation chain:
  * grad_weight: kappa = D + 8 (a chunk's dot product, the shuffle tree over
    a row's chunks, the four-corner combination);
  * grad_loc: kappa = D + S*G + 8 (the same, plus the sum over the S*G
    samples that share one location).
grad_feat sums one product per record of its feature row. Each product
carries three fp32 roundings (corner weight, times the sample weight, times
grad_out) and each addition one more, in any order, so a row of n records
has kappa = n + 2. Rows of the standard workloads hold few records and need
no such term. Tests that crowd thousands of samples onto a few pixels ask
for it ("grad_feat" in kind_names); n is then each row's own count, from
oracle.row_counts.
The oracle supplies M:
  * grad_weight: M is the oracle's grad_weight with |feat| and |grad_out|.
    Every product in it is then non-negative.
  * grad_loc: M comes from oracle.grad_loc_magnitude.
A dropped corner, a wrong sign or a swapped axis moves an element by about M
(by about M/n for a grad_feat row of n records), far beyond kappa*u*M.
For grad_feat, M is the oracle's grad_feat with |weights| and |grad_out|.
"""
from __future__ import annotations

import numpy as np
import torch

EPS32 = float(np.finfo(np.float32).eps)

TOL = {
    "f32": {"out": (1e-5, 1e-6), "grad_feat": (1e-4, 1e-6), "grad_loc": (1e-4, 1e-6),
            "grad_weight": (1e-4, 1e-6)},
    # fp16 features: the oracle reads the same fp16 values exactly widened and
    # the kernels compute in fp32, so the fp32 bounds apply.
    "f16": {"out": (1e-5, 1e-6), "grad_feat": (1e-4, 1e-6), "grad_loc": (1e-4, 1e-6),
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


U32 = 2.0 ** -24

# Share of a tensor's elements allowed outside the plain rtol/atol bound that
# pass only through the kappa*u*M term (the first sp4d_train run had 89 of
# 842,400 grad_loc elements there, 1.1e-4 of them), with a floor for small
# tensors.
PLAIN_EXCESS_SHARE = 5e-4
PLAIN_EXCESS_FLOOR = 8


def plain_excess_cap(size: int) -> int:
    return max(PLAIN_EXCESS_FLOOR, int(PLAIN_EXCESS_SHARE * size))


def plain_bound_excess(gpu: np.ndarray, ref: np.ndarray, rtol: float, atol: float, name: str = "") -> int:
    """Number of elements outside the plain |g-r| <= rtol*|r| + atol bound
    (before the kappa*u*M term); printed so a test log shows it."""
    n, msg = violations(gpu, ref, rtol, atol, name)
    print(f"{name}: {n}/{np.size(ref)} outside the plain bound" + (f" ({msg})" if n else ""))
    return n


def widened_violations(gpu: np.ndarray, ref: np.ndarray, rtol: float, atol: float, term, name: str = ""):
    """Messages for an output whose bound carries the kappa*u*M term `term`
    (an array of ref's size, or None for none): elements outside
    rtol*|ref| + atol + term, and more elements than plain_excess_cap
    outside the plain rtol*|ref| + atol bound."""
    msgs = []
    if term is not None:
        n_plain = plain_bound_excess(gpu, ref, rtol, atol, name)
        cap = plain_excess_cap(np.size(ref))
        if n_plain > cap:
            msgs.append(f"{name}: {n_plain} elements pass only through the kappa*u*M term (cap {cap})")
        atol = atol + np.reshape(term, np.shape(ref))
    n, msg = violations(gpu, ref, rtol, atol, name)
    if n:
        msgs.append(msg)
    return msgs


def conditioning_atol(inp, kind_names=("grad_loc", "grad_weight")):
    """Per-element kappa*u*M for grad_loc, grad_weight and, when asked,
    grad_feat (see the module doc)."""
    import oracle
    wl = inp.wl
    K, S = inp.spatial_shape.shape[0], inp.spatial_shape.shape[1]
    G = inp.weights.shape[-1]
    D = inp.feat.shape[-1] // G
    feat = inp.feat_numpy()
    afeat = (feat & np.uint16(0x7FFF)) if feat.dtype == np.uint16 else np.abs(feat)
    args = (inp.spatial_shape.numpy(), inp.level_start_index.numpy(), inp.loc.numpy(),
            inp.weights.numpy())
    go = inp.grad_out.numpy()
    res = {}
    if "grad_weight" in kind_names:
        _, _, m_gw = oracle.backward(afeat, *args, np.abs(go))
        res["grad_weight"] = (D + 8) * U32 * m_gw.astype(np.float64)
    if "grad_feat" in kind_names:
        n_row = oracle.row_counts(feat, *args).astype(np.float64)
        m_gf, _, _ = oracle.backward(feat, *args[:3], np.abs(inp.weights.numpy()), np.abs(go))
        res["grad_feat"] = (n_row[:, :, None] + 2) * U32 * m_gf.astype(np.float64)
    if "grad_loc" in kind_names:
        m_gl = oracle.grad_loc_magnitude(feat, *args, go)
        res["grad_loc"] = (D + S * G + 8) * U32 * m_gl.astype(np.float64)
    return res


def max_rel(gpu: np.ndarray, ref: np.ndarray, floor: float = 1e-3) -> float:
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), floor))) if g.size else 0.0
