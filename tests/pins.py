"""Pins of the CPU oracle: checks against facts fixed by the pages and by
arithmetic, not by the oracle itself.

Each ``pin_*`` function takes an :class:`oracle.Oracle` and raises
AssertionError when the oracle disagrees with a closed form, an exact integer
sum, a brute-force rational evaluation, an invariant, or a worked example
printed on the pages.  tests/test_oracle_pins.py runs them on the real oracle;
tests/test_oracle_mutants.py runs them on deliberately broken builds of the
oracle to show that a plausible mistake (a dropped term, a wrong sign, a
transposed index, a wrong scan direction) fails at least one pin.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np

from oracle import brute
from reduction_scan_primitives_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EULER_GAMMA = 0.57721566490153286060651209008240243104215933593992
U64 = 2.0 ** -53


def _np(t):
    return t.numpy() if hasattr(t, "numpy") else np.asarray(t)


def harmonic_closed_form(n: int) -> float:
    """H_n from the Euler-Maclaurin expansion (truncation error < 1/(240 n^8))."""
    return (math.log(n) + EULER_GAMMA + 1.0 / (2 * n) - 1.0 / (12 * n ** 2)
            + 1.0 / (120 * n ** 4) - 1.0 / (252 * n ** 6))


def pin_sum_harmonic(orc):
    """x[i] = fp32(1/(i+1)) sums to H_n (High-Performance Reduction Kernels
    README, 'Layout' section).  Each input carries a rounding error of at most
    half an fp32 ulp, so the fp64 sum of the rounded inputs must lie within
    2^-24 * H_n of the exact harmonic number, and within fp64 rounding of the
    correctly rounded sum (math.fsum) of the same fp32 values."""
    for n in (1, 2, 3, 4, 7, 10):
        x = _np(inputs.make((n,), "harmonic"))
        s, a = orc.sum1d(x)
        exact = sum((Fraction(1, i + 1) for i in range(n)), Fraction(0))
        assert abs(s - float(exact)) <= 2.0 ** -24 * float(exact) + 1e-15, (n, s, exact)
        assert a == s
    n = 1_000_000
    x = _np(inputs.make((n,), "harmonic"))
    s, a = orc.sum1d(x)
    h = harmonic_closed_form(n)
    assert abs(s - h) <= 2.0 ** -24 * h, (s, h)
    fs = math.fsum(x.astype(np.float64).tolist())
    assert abs(s - fs) <= 1e-12 * fs, (s, fs)
    assert a == s


def pin_sum_constant(orc):
    """A constant c summed n times is n*c.  fp32 c has 24 significant bits, so
    every partial k*c (k < 2^29) is exact in fp64 and the result is exact."""
    for c in (1.0, 0.5, -3.0, float(np.float32(0.1))):
        for n in (0, 1, 17, 1000, 100_003):
            x = np.full(n, c, dtype=np.float32)
            s, a = orc.sum1d(x)
            assert s == n * float(np.float32(c)), (c, n, s)
            assert a == n * abs(float(np.float32(c))), (c, n, a)


def pin_sum_integers(orc):
    """Small-integer inputs sum exactly: compare with an int64 sum."""
    for dist, n, seed in (("int:-8:8", 100_003, 5), ("int:-1:1", 1_000_000, 42), ("int:0:3", 777, 9)):
        x = _np(inputs.make((n,), dist, seed))
        s, a = orc.sum1d(x)
        xi = x.astype(np.int64)
        assert s == float(xi.sum()), (dist, s, xi.sum())
        assert a == float(np.abs(xi).sum())


def _mixed_values(rng, n):
    """Random fp32 values with mixed signs and exponents."""
    v = rng.standard_normal(n) * np.exp2(rng.integers(-6, 7, n))
    return v.astype(np.float32)


def pin_sum_bruteforce(orc):
    """Against an exact rational sum on tiny arrays.  A sequential fp64 sum of
    n terms is within (n-1) * 2^-53 * sum|x| of the exact value."""
    rng = np.random.default_rng(1234)
    for n in list(range(0, 13)) + [31, 64]:
        x = _mixed_values(rng, n)
        s, a = orc.sum1d(x)
        exact = brute.sum_exact(x.tolist())
        exact_abs = brute.sum_exact(abs(v) for v in x.tolist())
        assert abs(s - float(exact)) <= max(n - 1, 0) * U64 * float(exact_abs) + 1e-300, (n, s, exact)
        assert abs(a - float(exact_abs)) <= max(n - 1, 0) * U64 * float(exact_abs) + 1e-300


AXIS_SHAPES = [(1, 1, 1), (2, 3, 4), (3, 1, 5), (4, 5, 1), (1, 6, 3), (2, 0, 3), (0, 3, 2),
               (3, 7, 2), (2, 5, 3), (5, 2, 6)]


def pin_axis_bruteforce(orc):
    """out[o, i] = sum_r x[o, r, i] against exact rational sums written with
    their own index arithmetic (POPCORNBENCH trace l1_p47, problem statement:
    [batch, dim1, dim2] summed over dim 1)."""
    rng = np.random.default_rng(99)
    for (o, r, i) in AXIS_SHAPES:
        x = _mixed_values(rng, o * r * i)
        out, aout = orc.axis_sum(x, o, r, i)
        assert out.shape == (o, i)
        ex = brute.axis_sum_exact(x.tolist(), o, r, i)
        exa = brute.axis_sum_exact([abs(v) for v in x.tolist()], o, r, i)
        for a in range(o):
            for b in range(i):
                bound = max(r - 1, 0) * U64 * float(exa[a][b]) + 1e-300
                assert abs(out[a, b] - float(ex[a][b])) <= bound, ((o, r, i), a, b)
                assert abs(aout[a, b] - float(exa[a][b])) <= bound
        if r == 0:
            assert np.all(out == 0.0)


def pin_axis_integers_and_invariants(orc):
    """Exact on small integers (int64 reference over the same axis); inner == 1
    reduces each row like the 1D sum; outer == inner == 1 is the 1D sum; the
    positional variant agrees with the full one."""
    x = _np(inputs.make((3, 100, 7), "int:-8:8", 5))
    out, aout = orc.axis_sum(x, 3, 100, 7)
    xi = x.astype(np.int64)
    assert np.array_equal(out, xi.sum(axis=1).astype(np.float64))
    assert np.array_equal(aout, np.abs(xi).sum(axis=1).astype(np.float64))
    rng = np.random.default_rng(7)
    rows = _mixed_values(rng, 5 * 33).reshape(5, 33)
    out, _ = orc.axis_sum(rows, 5, 33, 1)
    for k in range(5):
        assert out[k, 0] == orc.sum1d(rows[k])[0]
    flat = _mixed_values(rng, 50)
    assert orc.axis_sum(flat, 1, 50, 1)[0][0, 0] == orc.sum1d(flat)[0]
    x = _mixed_values(rng, 4 * 9 * 6)
    full, fabs_ = orc.axis_sum(x, 4, 9, 6)
    pos = np.array([0, 5, 6, 13, 23, 17], dtype=np.int64)
    at, at_abs = orc.axis_sum_at(x, 4, 9, 6, pos)
    assert np.array_equal(at, full.reshape(-1)[pos])
    assert np.array_equal(at_abs, fabs_.reshape(-1)[pos])


def pin_scan_worked_examples(orc):
    """The worked examples of the POPCORNBENCH trace l1_p91 (reverse cumsum):
    [1..8] -> [36, 35, 33, 30, 26, 21, 15, 8]; [a, b, c, d] -> [a+b+c+d,
    b+c+d, c+d, d]."""
    with open(os.path.join(GOLDEN, "rcumsum_worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        x = np.asarray(c["x"], dtype=np.float32)
        y, ay = orc.reverse_cumsum(x, 1, x.size)
        assert y.reshape(-1).tolist() == [float(v) for v in c["y"]], (c, y)
        assert ay.reshape(-1).tolist() == [float(v) for v in c["y"]]


def pin_scan_bruteforce(orc):
    """Against the O(N^2) definition (exact rationals) on tiny shapes, plus:
    the last column equals x exactly (a suffix of one term), the first column
    is the row sum."""
    rng = np.random.default_rng(5)
    for rows, n in ((1, 1), (1, 2), (2, 3), (3, 5), (2, 8), (4, 1), (1, 13), (3, 4)):
        x = _mixed_values(rng, rows * n)
        y, ay = orc.reverse_cumsum(x, rows, n)
        ex = brute.reverse_cumsum_exact(x.tolist(), rows, n)
        exa = brute.reverse_cumsum_exact([abs(v) for v in x.tolist()], rows, n)
        for a in range(rows):
            for j in range(n):
                bound = (n - j) * U64 * float(exa[a][j]) + 1e-300
                assert abs(y[a, j] - float(ex[a][j])) <= bound, (rows, n, a, j)
                assert abs(ay[a, j] - float(exa[a][j])) <= bound
        xr = x.reshape(rows, n).astype(np.float64)
        assert np.array_equal(y[:, -1], xr[:, -1])
        for a in range(rows):
            s, sa = orc.sum1d(x.reshape(rows, n)[a])
            assert abs(y[a, 0] - s) <= n * U64 * sa + 1e-300


def pin_scan_integers(orc):
    """Exact on small integers: the result equals flip-cumsum-flip in int64
    (the reference expression of the POPCORNBENCH trace l1_p91), and
    consecutive differences give back x."""
    x = _np(inputs.make((6, 301), "int:0:3", 3))
    y, ay = orc.reverse_cumsum(x, 6, 301)
    xi = x.astype(np.int64)
    ref = np.flip(np.cumsum(np.flip(xi, axis=1), axis=1), axis=1)
    assert np.array_equal(y, ref.astype(np.float64))
    assert np.array_equal(ay, ref.astype(np.float64))
    assert np.array_equal(y[:, :-1] - y[:, 1:], xi[:, :-1].astype(np.float64))
    x = _np(inputs.make((2, 257), "int:-8:8", 4))
    y, ay = orc.reverse_cumsum(x, 2, 257)
    xi = x.astype(np.int64)
    assert np.array_equal(y, np.flip(np.cumsum(np.flip(xi, 1), 1), 1).astype(np.float64))
    assert np.array_equal(ay, np.flip(np.cumsum(np.flip(np.abs(xi), 1), 1), 1).astype(np.float64))


CUMSUM_SHAPES = [(1, 1, 1), (1, 8, 1), (2, 5, 3), (3, 4, 2), (1, 7, 4), (2, 1, 5), (4, 6, 1)]
MODES = [(False, False), (False, True), (True, False), (True, True)]


def pin_cumsum_bruteforce(orc):
    """Forward / reverse, inclusive / exclusive cumulative sums along the middle
    axis of [outer, N, inner] against exact rational sums, one per output,
    written with their own index ranges (the POPCORNBENCH trace l1_p91
    discusses the reverse scan along dim 1 and other dims)."""
    rng = np.random.default_rng(21)
    for (o, n, i) in CUMSUM_SHAPES:
        x = _mixed_values(rng, o * n * i)
        for rev, exc in MODES:
            y, ay = orc.cumsum(x, o, n, i, rev, exc)
            ex = brute.cumsum_exact(x.tolist(), o, n, i, rev, exc)
            exa = brute.cumsum_exact([abs(v) for v in x.tolist()], o, n, i, rev, exc)
            for a in range(o):
                for j in range(n):
                    for b in range(i):
                        bound = n * U64 * float(exa[a][j][b]) + 1e-300
                        assert abs(y[a, j, b] - float(ex[a][j][b])) <= bound, ((o, n, i), rev, exc, a, j, b)
                        assert abs(ay[a, j, b] - float(exa[a][j][b])) <= bound


def pin_cumsum_worked_examples(orc):
    """The hand traces of the POPCORNBENCH trace l1_p91: reverse inclusive
    [1..8] -> [36, ..., 8] and forward exclusive [1..8] -> [0, 1, 3, ..., 28]."""
    with open(os.path.join(GOLDEN, "exclusive_scan_worked_example.json")) as f:
        cases = json.load(f)["cases"]
    with open(os.path.join(GOLDEN, "rcumsum_worked_examples.json")) as f:
        cases += [dict(c, reverse=True, exclusive=False) for c in json.load(f)["cases"]]
    for c in cases:
        x = np.asarray(c["x"], dtype=np.float32)
        y, _ = orc.cumsum(x, 1, x.size, 1, c["reverse"], c["exclusive"])
        assert y.reshape(-1).tolist() == [float(v) for v in c["y"]], (c, y)


def pin_cumsum_integers(orc):
    """Exact on small integers against int64 cumsum written with numpy: forward
    = cumsum, reverse = flip-cumsum-flip, exclusive = the inclusive result
    shifted by one; the reverse inclusive case equals the reverse-cumsum
    routine's result."""
    x = _np(inputs.make((3, 50, 4), "int:-8:8", 6))
    xi = x.astype(np.int64)
    fwd = np.cumsum(xi, axis=1)
    rev = np.flip(np.cumsum(np.flip(xi, 1), axis=1), 1)
    zero = np.zeros((3, 1, 4), np.int64)
    want = {(False, False): fwd, (True, False): rev,
            (False, True): np.concatenate([zero, fwd[:, :-1]], axis=1),
            (True, True): np.concatenate([rev[:, 1:], zero], axis=1)}
    for (r, e), ref in want.items():
        y, ay = orc.cumsum(x, 3, 50, 4, r, e)
        assert np.array_equal(y, ref.astype(np.float64)), (r, e)
    x2 = _np(inputs.make((5, 77), "int:0:3", 8))
    y, _ = orc.cumsum(x2, 5, 77, 1, True, False)
    assert np.array_equal(y[:, :, 0], orc.reverse_cumsum(x2, 5, 77)[0])


OP_SHAPES = [(1, 1, 1), (2, 5, 3), (3, 1, 4), (1, 9, 1), (4, 6, 2)]


def pin_reduce_ops_bruteforce(orc):
    """Max and min against Python's max()/min() (exact), mean against the exact
    rational mean, the norm squared against the exact rational sum of squares
    (the "Seven-step reduction" page lists sum, max and the L2 norm as the same
    reduction pattern)."""
    rng = np.random.default_rng(31)
    for (o, r, i) in OP_SHAPES:
        x = _mixed_values(rng, o * r * i)
        for op in ("mean", "max", "min", "norm"):
            out, sc = orc.reduce_op(x, o, r, i, op)
            ex = brute.reduce_op_exact(x.tolist(), o, r, i, op)
            for a in range(o):
                for b in range(i):
                    if op in ("max", "min"):
                        assert out[a, b] == float(ex[a][b]), (op, (o, r, i), a, b)
                    elif op == "mean":
                        scale = sum(abs(float(x[(a * r + k) * i + b])) for k in range(r))
                        assert abs(out[a, b] - float(ex[a][b])) <= r * U64 * scale / r + 1e-300, (op, a, b)
                    else:
                        want = float(ex[a][b])
                        assert abs(out[a, b] ** 2 - want) <= (r + 2) * U64 * want + 1e-300, (op, a, b)


def pin_reduce_ops_closed_forms(orc):
    """Closed forms: the mean of 1..n is (n+1)/2; a constant c has mean c,
    max = min = c and norm |c| sqrt(n); the norms of (3, 4) and (1, 2, 2) are
    5 and 3; NaN propagates through max and min; empty axes give -inf, +inf,
    NaN and 0."""
    n = 1001
    x = np.arange(1, n + 1, dtype=np.float32)
    assert orc.reduce_op(x, 1, n, 1, "mean")[0][0, 0] == (n + 1) / 2
    assert orc.reduce_op(x, 1, n, 1, "max")[0][0, 0] == n
    assert orc.reduce_op(x, 1, n, 1, "min")[0][0, 0] == 1
    c = np.full(400, -2.5, dtype=np.float32)
    assert orc.reduce_op(c, 1, 400, 1, "mean")[0][0, 0] == -2.5
    assert orc.reduce_op(c, 1, 400, 1, "norm")[0][0, 0] == 2.5 * 20.0
    assert orc.reduce_op(np.array([3, 4], np.float32), 1, 2, 1, "norm")[0][0, 0] == 5.0
    assert orc.reduce_op(np.array([1, 2, 2], np.float32), 1, 3, 1, "norm")[0][0, 0] == 3.0
    y = np.array([1.0, np.nan, 7.0], np.float32)
    assert np.isnan(orc.reduce_op(y, 1, 3, 1, "max")[0][0, 0])
    assert np.isnan(orc.reduce_op(y, 1, 3, 1, "min")[0][0, 0])
    e = np.zeros(0, np.float32)
    assert orc.reduce_op(e, 2, 0, 3, "max")[0].tolist() == [[-np.inf] * 3] * 2
    assert orc.reduce_op(e, 2, 0, 3, "min")[0].tolist() == [[np.inf] * 3] * 2
    assert np.isnan(orc.reduce_op(e, 1, 0, 1, "mean")[0][0, 0])
    assert orc.reduce_op(e, 1, 0, 1, "norm")[0][0, 0] == 0.0
    # Strided axis with integers: exact against int64 arithmetic.
    z = _np(inputs.make((3, 40, 5), "int:-8:8", 12))
    zi = z.astype(np.int64)
    assert np.array_equal(orc.reduce_op(z, 3, 40, 5, "max")[0], zi.max(axis=1).astype(np.float64))
    assert np.array_equal(orc.reduce_op(z, 3, 40, 5, "min")[0], zi.min(axis=1).astype(np.float64))
    # The sum of squares of small integers is exact, and sqrt is correctly rounded.
    assert np.array_equal(orc.reduce_op(z, 3, 40, 5, "norm")[0],
                          np.sqrt((zi * zi).sum(axis=1).astype(np.float64)))


ALL_PINS = [pin_sum_harmonic, pin_sum_constant, pin_sum_integers, pin_sum_bruteforce,
            pin_axis_bruteforce, pin_axis_integers_and_invariants, pin_scan_worked_examples,
            pin_scan_bruteforce, pin_scan_integers, pin_cumsum_bruteforce, pin_cumsum_worked_examples,
            pin_cumsum_integers, pin_reduce_ops_bruteforce, pin_reduce_ops_closed_forms]
