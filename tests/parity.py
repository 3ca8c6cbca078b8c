"""Helpers for comparing the CUDA path with the oracle, element by element.

Acceptance per output (the bound the library documents):
    |gpu - ref| <= 1e-5 * sum|x over that output's terms| + 1e-6
Non-finite references: a NaN reference needs a NaN result, an infinite one
the same infinity.  Integer-valued inputs must match exactly.
"""
import numpy as np

import oracle


def to_np(t):
    if hasattr(t, "detach"):
        t = t.detach()
        if t.device.type != "cpu":
            t = t.cpu()
        return t.numpy()
    return np.asarray(t)


def assert_close(gpu, ref, abs_ref, what=""):
    g = np.asarray(to_np(gpu), dtype=np.float64).reshape(-1)
    r = np.asarray(ref, dtype=np.float64).reshape(-1)
    a = np.asarray(abs_ref, dtype=np.float64).reshape(-1)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    fin = np.isfinite(r)
    tol = oracle.tolerance(a)
    err = np.abs(g - r)
    bad = fin & ~(err <= tol)
    if bad.any():
        k = int(np.flatnonzero(bad)[0])
        worst = int(np.argmax(np.where(fin, err / tol, 0)))
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{g.size} outputs out of tolerance; first at {k}: gpu={g[k]!r} "
            f"ref={r[k]!r} tol={tol[k]:.3e}; worst ratio {err[worst] / tol[worst]:.3f} at {worst}")
    nan_ref = np.isnan(r)
    assert np.all(np.isnan(g[nan_ref])), f"{what}: NaN expected"
    inf_ref = np.isinf(r)
    assert np.array_equal(g[inf_ref], r[inf_ref]), f"{what}: infinity expected"


def assert_exact(gpu, ref, what=""):
    g = np.asarray(to_np(gpu), dtype=np.float64).reshape(-1)
    r = np.asarray(ref, dtype=np.float64).reshape(-1)
    diff = np.flatnonzero(g != r)
    assert diff.size == 0, f"{what}: {diff.size} outputs differ, first at {diff[0]}: {g[diff[0]]} vs {r[diff[0]]}"


def error_ratio(gpu, ref, abs_ref):
    """max |gpu - ref| / (2^-24 * sum|x|): the error in units of fp32 rounding
    of the absolute scale (informational; a tree of depth d stays below ~d)."""
    g = np.asarray(to_np(gpu), dtype=np.float64).reshape(-1)
    r = np.asarray(ref, dtype=np.float64).reshape(-1)
    a = np.asarray(abs_ref, dtype=np.float64).reshape(-1)
    m = a > 0
    if not m.any():
        return 0.0
    return float(np.max(np.abs(g[m] - r[m]) / (2.0 ** -24 * a[m])))


def bitwise_equal(a, b):
    import torch
    return torch.equal(a.view(torch.int32), b.view(torch.int32))
