"""Pure-Python brute force for tiny inputs (test infrastructure only).

These loops restate the definitions a second, independent way (Python floats,
with exact rational arithmetic where asked) so the C oracle can be checked
against something that is not itself.  Use only for tiny shapes.
"""
from fractions import Fraction


def sum_exact(values):
    """Exact rational sum of float values (each float is an exact rational)."""
    total = Fraction(0)
    for v in values:
        total += Fraction(float(v))
    return total


def axis_sum_exact(flat, outer, reduce, inner):
    """Exact out[o][i] = sum_r x[o, r, i], index arithmetic written out."""
    out = []
    for o in range(outer):
        row = []
        for i in range(inner):
            terms = [flat[(o * reduce + r) * inner + i] for r in range(reduce)]
            row.append(sum_exact(terms))
        out.append(row)
    return out


def reverse_cumsum_exact(flat, rows, n):
    """Exact y[i][j] = sum over k from j to n-1 of x[i, k] (O(n^2) per row)."""
    out = []
    for i in range(rows):
        row = []
        for j in range(n):
            row.append(sum_exact(flat[i * n + k] for k in range(j, n)))
        out.append(row)
    return out


def cumsum_exact(flat, outer, n, inner, reverse=False, exclusive=False):
    """Exact y[o][j][i] = sum of x[o, k, i] over k <= j (forward) or k >= j
    (reverse), with k == j left out when exclusive; one sum per output."""
    out = []
    for o in range(outer):
        plane = []
        for j in range(n):
            if reverse:
                ks = range(j + 1 if exclusive else j, n)
            else:
                ks = range(0, j if exclusive else j + 1)
            plane.append([sum_exact(flat[(o * n + k) * inner + i] for k in ks) for i in range(inner)])
        out.append(plane)
    return out


def reduce_op_exact(flat, outer, reduce, inner, op):
    """mean / max / min / squared norm of x[o, :, i] with Python built-ins and
    exact rationals (the norm is returned squared, exactly)."""
    out = []
    for o in range(outer):
        row = []
        for i in range(inner):
            vals = [flat[(o * reduce + r) * inner + i] for r in range(reduce)]
            if op == "mean":
                row.append(sum_exact(vals) / len(vals) if vals else None)
            elif op == "max":
                row.append(max(vals) if vals else float("-inf"))
            elif op == "min":
                row.append(min(vals) if vals else float("inf"))
            else:
                total = Fraction(0)
                for v in vals:
                    total += Fraction(float(v)) * Fraction(float(v))
                row.append(total)
        out.append(row)
    return out
