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


def assert_op_close(gpu, ref, scale, op, count, what):
    """mean: (1e-5 sum|x| + 1e-6) / count plus one fp32 rounding; norm:
    1e-5 norm + 1e-6; max and min: exact (NaN for NaN)."""
    g = np.asarray(to_np(gpu), np.float64).reshape(-1)
    r = np.asarray(ref, np.float64).reshape(-1)
    sc = np.asarray(scale, np.float64).reshape(-1)
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(g), nan), f"{what}: NaN pattern differs"
    g, r, sc = g[~nan], r[~nan], sc[~nan]
    if op in ("max", "min"):
        bad = np.flatnonzero(g != r)
        assert bad.size == 0, f"{what}: {bad.size} differ, first {bad[0]}: {g[bad[0]]} vs {r[bad[0]]}"
        return
    if op == "mean":
        tol = (1e-5 * sc + 1e-6) / max(count, 1) + 2.0 ** -24 * np.abs(r)
    else:
        tol = 1e-5 * r + 1e-6
    fin = np.isfinite(r)
    bad = np.flatnonzero(fin & ~(np.abs(g - r) <= tol))
    assert bad.size == 0, f"{what}: {bad.size} out of tolerance, first {bad[0]}: {g[bad[0]]} vs {r[bad[0]]}"
    assert np.array_equal(g[~fin], r[~fin])
