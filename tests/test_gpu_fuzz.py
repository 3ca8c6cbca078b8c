"""Seeded random cases across every entry point and strategy, against the
oracle (GPU).

Each case draws a shape (1 to 3 dims, total size log-uniform), an axis, the scan
direction and exclusivity, a pointer offset of 0-3 floats, and the library
options that steer the kernel choice (reduce-axis split, column-kernel and
column-scan shapes, the narrow-row and narrow-plane forms, the row-scan
strategy), so the
many paths and their ragged edges meet inputs nobody picked by hand.  A
failure names the case's parameters."""
import numpy as np
import pytest

import oracle
from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import assert_close, assert_exact, assert_op_close
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu
CHUNKS, PER_CHUNK = 12, 40


def draw_shape(rng, max_total):
    """Total size log-uniform in [1, max_total], split over 1-3 dims at random."""
    nd = int(rng.integers(1, 4))
    log_total = rng.uniform(0, np.log(max_total))
    parts = rng.dirichlet(np.ones(nd)) * log_total
    return tuple(max(1, int(np.exp(p))) for p in parts)


def draw_case(rng):
    kind = str(rng.choice(["sum", "reduce", "scan", "scan"]))
    shape = draw_shape(rng, 3_000_000 if kind != "scan" else 2_000_000)
    case = dict(kind=kind, shape=shape, dim=int(rng.integers(0, len(shape))),
                op=str(rng.choice(["sum", "mean", "max", "min", "norm"])),
                reverse=bool(rng.integers(0, 2)), exclusive=bool(rng.integers(0, 2)),
                offset=int(rng.integers(0, 4)), dist=str(rng.choice(["uniform_pm1", "normal", "int:-8:8"])),
                seed=int(rng.integers(0, 1 << 30)),
                split=int(rng.choice([0, 0, 0, 1, 2, 7, 64])),
                cols_variant=int(rng.choice([-1, -1, 0, 1, 2, 3, 4, 5, 6, 7, 8, 9])),
                scan_cols_variant=int(rng.choice([-1, -1, 0, 1, 2, 3, 4, 5, 6, 7, 8, 9])),
                strategy=int(rng.choice([0, 0, 1, 2, 3, 4])))
    if case["dist"] == "int:-8:8" and case["kind"] == "scan":
        case["dist"] = "int:0:3"  # partial sums stay exact in fp32
    return case


def run_case(c):
    L.set_option(L.OPT_AXIS_SPLIT, c["split"])
    L.set_option(L.OPT_COLS_VARIANT, c["cols_variant"])
    L.set_option(L.OPT_SCAN_COLS_VARIANT, c["scan_cols_variant"])
    L.set_option(L.OPT_SCAN_STRATEGY, c["strategy"])
    x = inputs.make(c["shape"], c["dist"], c["seed"])
    xd = on_device(x, c["offset"])
    what = str(c)
    # Integer inputs sum exactly while every partial sum stays below 2^24.
    exact_terms = lambda terms: c["dist"].startswith("int") and terms * 8 < (1 << 24)  # noqa: E731
    if c["kind"] == "sum":
        got = L.reduce_sum_f32(xd.reshape(-1)).cpu().numpy().reshape(-1)
        ref, scale = oracle.sum1d(x.numpy().reshape(-1))
        if exact_terms(x.numel()):
            assert_exact(got, [ref], what)
        else:
            assert_close(got, [ref], [scale], what)
        return
    o, n, i = L.canonical_axis(c["shape"], c["dim"])
    exact = exact_terms(n)
    if c["kind"] == "reduce":
        got = L.reduce_axis_op_f32(xd, c["dim"], c["op"]).cpu().numpy().reshape(-1)
        if c["op"] == "sum":
            ref, scale = oracle.axis_sum(x.numpy(), o, n, i)
            if exact:
                assert_exact(got, ref, what)
            else:
                assert_close(got, ref, scale, what)
        else:
            ref, scale = oracle.reduce_op(x.numpy(), o, n, i, c["op"])
            assert_op_close(got, ref, scale, c["op"], n, what)
        return
    got = L.cumsum_f32(xd, c["dim"], reverse=c["reverse"], exclusive=c["exclusive"]).cpu().numpy().reshape(-1)
    ref, scale = oracle.cumsum(x.numpy(), o, n, i, c["reverse"], c["exclusive"])
    if exact:
        assert_exact(got, ref.reshape(-1), what)
    else:
        assert_close(got, ref.reshape(-1), scale.reshape(-1), what)


@pytest.mark.parametrize("chunk", range(CHUNKS))
def test_random_cases(chunk):
    rng = np.random.default_rng(20261202 + chunk)
    for _ in range(PER_CHUNK):
        run_case(draw_case(rng))
    L.check()
