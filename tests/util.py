"""Helpers shared by the parity tests: device transfer and the tolerance checks.

Tolerances (from the workload specification): a floating-point projection output
must satisfy |y_gpu − y_ref| ≤ 1e-3 · e with e = Σ_c |w||x| (the oracle's error
scale of that element); RMSNorm scales inv within 1e-4 relative.  Derived outputs
get the bound that follows from these by first-order propagation (stated where
used)."""
from __future__ import annotations

import numpy as np

TOL = 1e-3          # projections: |Δ| ≤ TOL · Σ|w||x|
NORM_TOL = 1e-4     # RMSNorm scales: relative


def cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    return t.detach().cpu().numpy()


def check_proj(got, ref, e, tol=TOL, what="projection", extra=0.0):
    """|got − ref| ≤ tol·e + extra elementwise; reports the worst ratio."""
    got = np.asarray(got, np.float64).reshape(np.shape(ref))
    ref = np.asarray(ref, np.float64)
    e = np.asarray(e, np.float64).reshape(ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    lim = tol * e + extra + 1e-30
    ratio = float((err / lim).max())
    assert np.all(err <= lim), f"{what}: max |Δ|/limit = {ratio:.3g}"
    return float((err / np.maximum(e, 1e-30)).max())


def check_relu2(got, y_ref, e_y, tol=TOL, what="relu²"):
    """u = relu²(y): with |Δy| ≤ d = tol·e, |Δu| ≤ 2|y|·d + d²."""
    y_ref = np.asarray(y_ref, np.float64)
    d = tol * np.asarray(e_y, np.float64).reshape(y_ref.shape)
    u_ref = np.maximum(y_ref, 0) ** 2
    got = np.asarray(got, np.float64).reshape(u_ref.shape)
    err = np.abs(got - u_ref)
    lim = 2 * np.abs(y_ref) * d + d * d + 1e-30
    assert np.all(err <= lim), f"{what}: max |Δ|/limit = {(err / lim).max():.3g}"


def check_rel(got, ref, rel, what, abs_=0.0):
    got = np.asarray(got, np.float64).reshape(np.shape(ref))
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    lim = rel * np.abs(ref) + abs_
    assert np.all(err <= lim), f"{what}: max rel err {(err / np.maximum(np.abs(ref), 1e-300)).max():.3g}"
