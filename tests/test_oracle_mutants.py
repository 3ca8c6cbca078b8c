"""Plant plausible mistakes in copies of the oracle (on the CPU) and check
that the pins catch every one of them.  The real oracle.c is never changed."""
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild
import pins

# (name, function whose body is edited, text to replace, replacement)
MUTANTS = [
    ("sum_drops_last_term", "oracle_sum", "i < n; ++i", "i + 1 < n; ++i"),
    ("sum_drops_first_term", "oracle_sum", "int64_t i = 0;", "int64_t i = 1;"),
    ("sum_wrong_sign", "oracle_sum", "s += v;", "s -= v;"),
    ("sum_abs_not_abs", "oracle_sum", "a += fabs(v);", "a += v;"),
    ("axis_transposed_index", "oracle_axis_sum", "x[(o * reduce + r) * inner + i]",
     "x[(o * inner + i) * reduce + r]"),
    ("axis_wrong_output_index", "oracle_axis_sum", "out[o * inner + i] = s;", "out[i * outer + o] = s;"),
    ("axis_drops_last_row", "oracle_axis_sum", "r < reduce", "r + 1 < reduce"),
    ("axis_abs_not_abs", "oracle_axis_sum", "a += fabs(v);", "a += v;"),
    ("scan_forward_direction", "oracle_reverse_cumsum", "for (int64_t j = N - 1; j >= 0; --j)",
     "for (int64_t j = 0; j < N; ++j)"),
    ("scan_exclusive", "oracle_reverse_cumsum", "y[i * N + j] = acc;", "y[i * N + j] = acc - v;"),
    ("scan_skips_last_column", "oracle_reverse_cumsum", "j = N - 1;", "j = N - 2;"),
    ("scan_no_row_reset", "oracle_reverse_cumsum", "double acc = 0.0;\n", ""),
    ("scan_abs_wrong", "oracle_reverse_cumsum", "acc_abs += fabs(v);", "acc_abs += v;"),
    ("at_swapped_position", "oracle_axis_sum_at", "int64_t o = pos[k] / inner;",
     "int64_t o = pos[k] % inner;"),
    ("cumsum_direction_ignored", "oracle_cumsum", "const int64_t j = reverse ? N - 1 - step : step;",
     "const int64_t j = step;"),
    ("cumsum_direction_swapped", "oracle_cumsum", "const int64_t j = reverse ? N - 1 - step : step;",
     "const int64_t j = reverse ? step : N - 1 - step;"),
    ("cumsum_exclusive_ignored", "oracle_cumsum", "if (exclusive) {", "if (0) {"),
    ("cumsum_wrong_index", "oracle_cumsum", "const int64_t idx = (o * N + j) * inner + i;",
     "const int64_t idx = (o * inner + i) * N + j;"),
    ("op_max_is_min", "oracle_reduce_op", "else if (v > acc) acc = v;", "else if (v < acc) acc = v;"),
    ("op_nan_dropped", "oracle_reduce_op", "if (isnan(v) || isnan(acc)) acc = NAN;\n          else if (v > acc)",
     "if (0) acc = NAN;\n          else if (v > acc)"),
    ("op_mean_not_divided", "oracle_reduce_op", "res = reduce > 0 ? acc / (double)reduce : NAN;",
     "res = reduce > 0 ? acc : NAN;"),
    ("op_norm_no_sqrt", "oracle_reduce_op", "if (op == 4) res = sqrt(acc);", "if (op == 4) res = acc;"),
    ("op_norm_abs_not_square", "oracle_reduce_op", "acc += v * v;", "acc += fabs(v);"),
    ("op_wrong_index", "oracle_reduce_op", "x[(o * reduce + r) * inner + i]", "x[(o * inner + i) * reduce + r]"),
    ("cumsum_no_reset", "oracle_cumsum", "      double acc = 0.0;\n      double acc_abs = 0.0;\n      for (int64_t step",
     "      double acc_abs = 0.0;\n      for (int64_t step"),
]


def _mutate(src, func, old, new):
    start = src.index(f"void {func}(")
    body = src[start:]
    assert old in body, (func, old)
    return src[:start] + body.replace(old, new, 1)


def _hoist_acc(src):
    # "scan_no_row_reset" removes the per-row reset; declare the accumulator
    # once per call instead so the mutant still compiles.
    return src.replace("void oracle_reverse_cumsum(const float* x, int64_t rows, int64_t N, double* y,\n"
                       "                           double* abs_y) {\n",
                       "void oracle_reverse_cumsum(const float* x, int64_t rows, int64_t N, double* y,\n"
                       "                           double* abs_y) {\n  double acc = 0.0;\n", 1)


@pytest.mark.parametrize("name,func,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, func, old, new):
    with open(obuild.SRC) as f:
        src = f.read()
    mutated = _mutate(src, func, old, new)
    if name == "scan_no_row_reset":
        mutated = _hoist_acc(mutated)
    if name == "cumsum_no_reset":
        mutated = mutated.replace("                   int exclusive, double* y, double* abs_y) {\n",
                                  "                   int exclusive, double* y, double* abs_y) {\n  double acc = 0.0;\n", 1)
    assert mutated != src
    csrc = tmp_path / "oracle_mutant.c"
    csrc.write_text(mutated)
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", *obuild.CFLAGS, "-I", obuild.HERE, "-o", str(lib), str(csrc), "-lm"],
                   check=True)
    orc = oracle.Oracle(str(lib))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
