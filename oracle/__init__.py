"""The CPU oracle: plain fp64 definitions of the three primitives.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library and its binding never import it, and it never imports them.

Functions take numpy float32 arrays (contiguous, host memory) and return fp64
results together with the companion sum of |x| over the same terms, which
scales the acceptance tolerance ``|gpu - ref| <= 1e-5 * sum|x| + 1e-6``.

Parity status: every function here is pinned (closed forms, exact integer
sums, brute force on tiny shapes, worked examples printed on the pages) in
tests/test_oracle_pins.py; nothing is "parity unpinned".
"""
import ctypes

import numpy as np

from . import build as _build

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_dp = ctypes.POINTER(ctypes.c_double)


def _as_f32(x):
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError(f"oracle expects float32 input, got {x.dtype}")
    return x.reshape(-1)


class Oracle:
    """ctypes view of one build of oracle.c (the default one, or a test build)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_sum.argtypes = [_f32p, _i64, _dp, _dp]
        lib.oracle_sum.restype = None
        lib.oracle_axis_sum.argtypes = [_f32p, _i64, _i64, _i64, _f64p, _f64p]
        lib.oracle_axis_sum.restype = None
        lib.oracle_reverse_cumsum.argtypes = [_f32p, _i64, _i64, _f64p, _f64p]
        lib.oracle_reverse_cumsum.restype = None
        lib.oracle_axis_sum_at.argtypes = [_f32p, _i64, _i64, _i64, _i64p, _i64, _f64p, _f64p]
        lib.oracle_axis_sum_at.restype = None
        lib.oracle_cumsum.argtypes = [_f32p, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _f64p, _f64p]
        lib.oracle_cumsum.restype = None
        lib.oracle_reduce_op.argtypes = [_f32p, _i64, _i64, _i64, ctypes.c_int, _f64p, _f64p]
        lib.oracle_reduce_op.restype = None
        self._lib = lib
        self.path = lib_path

    def sum1d(self, x):
        """(sum, sum|x|) of a float32 array, sequential fp64, left to right."""
        x = _as_f32(x)
        s = ctypes.c_double()
        a = ctypes.c_double()
        self._lib.oracle_sum(x, x.size, ctypes.byref(s), ctypes.byref(a))
        return s.value, a.value

    def axis_sum(self, x, outer, reduce, inner):
        """(out, abs_out), each fp64 [outer, inner]: sum over r of x[o, r, i]."""
        x = _as_f32(x)
        if x.size != outer * reduce * inner:
            raise ValueError("size mismatch")
        out = np.empty(outer * inner, np.float64)
        abs_out = np.empty(outer * inner, np.float64)
        self._lib.oracle_axis_sum(x, outer, reduce, inner, out, abs_out)
        return out.reshape(outer, inner), abs_out.reshape(outer, inner)

    def axis_sum_at(self, x, outer, reduce, inner, positions):
        """Axis sum at flat output positions p = o*inner + i (same definition)."""
        x = _as_f32(x)
        if x.size != outer * reduce * inner:
            raise ValueError("size mismatch")
        pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64).reshape(-1))
        if pos.size and (pos.min() < 0 or pos.max() >= outer * inner):
            raise ValueError("position out of range")
        out = np.empty(pos.size, np.float64)
        abs_out = np.empty(pos.size, np.float64)
        self._lib.oracle_axis_sum_at(x, outer, reduce, inner, pos, pos.size, out, abs_out)
        return out, abs_out

    def reverse_cumsum(self, x, rows, N):
        """(y, abs_y), each fp64 [rows, N]: y[i, j] = sum_{k >= j} x[i, k]."""
        x = _as_f32(x)
        if x.size != rows * N:
            raise ValueError("size mismatch")
        y = np.empty(rows * N, np.float64)
        abs_y = np.empty(rows * N, np.float64)
        self._lib.oracle_reverse_cumsum(x, rows, N, y, abs_y)
        return y.reshape(rows, N), abs_y.reshape(rows, N)


    def cumsum(self, x, outer, N, inner, reverse=False, exclusive=False):
        """(y, abs_y), each fp64 [outer, N, inner]: cumulative sum along the middle
        axis, forward (k <= j) or reverse (k >= j), inclusive or exclusive."""
        x = _as_f32(x)
        if x.size != outer * N * inner:
            raise ValueError("size mismatch")
        y = np.empty(outer * N * inner, np.float64)
        abs_y = np.empty(outer * N * inner, np.float64)
        self._lib.oracle_cumsum(x, outer, N, inner, int(bool(reverse)), int(bool(exclusive)), y, abs_y)
        return y.reshape(outer, N, inner), abs_y.reshape(outer, N, inner)


    OPS = {"mean": 1, "max": 2, "min": 3, "norm": 4}

    def reduce_op(self, x, outer, reduce, inner, op):
        """(out, scale), each fp64 [outer, inner]: mean / max / min / norm of
        x[o, :, i]; scale is sum|x| (mean) or sum x^2 (norm), 0 otherwise."""
        x = _as_f32(x)
        if x.size != outer * reduce * inner:
            raise ValueError("size mismatch")
        out = np.empty(outer * inner, np.float64)
        sc = np.empty(outer * inner, np.float64)
        self._lib.oracle_reduce_op(x, outer, reduce, inner, self.OPS[op], out, sc)
        return out.reshape(outer, inner), sc.reshape(outer, inner)


_default = None


def default() -> Oracle:
    """The oracle built from oracle/oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def sum1d(x):
    return default().sum1d(x)


def axis_sum(x, outer, reduce, inner):
    return default().axis_sum(x, outer, reduce, inner)


def axis_sum_at(x, outer, reduce, inner, positions):
    return default().axis_sum_at(x, outer, reduce, inner, positions)


def reverse_cumsum(x, rows, N):
    return default().reverse_cumsum(x, rows, N)


def cumsum(x, outer, N, inner, reverse=False, exclusive=False):
    return default().cumsum(x, outer, N, inner, reverse, exclusive)


def reduce_op(x, outer, reduce, inner, op):
    return default().reduce_op(x, outer, reduce, inner, op)


def tolerance(abs_scale):
    """Per-element acceptance bound 1e-5 * sum|x| + 1e-6 (fp64)."""
    return 1e-5 * np.asarray(abs_scale, dtype=np.float64) + 1e-6
