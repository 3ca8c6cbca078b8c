"""Narrow planes of 2 to 32 columns read flat as segmented class runs (GPU):
[outer, N, P] scanned or reduced along N by k_planes, which reads each tile of
the flat array into shared memory and scans runs of whole rows per thread, the
column classes fixed and the segments restarting at plane boundaries; scans of
other column counts up to 128 by k_planes_cg, one column group (a float4,
float2 or float) of a run of 9, 17 or 33 rows per thread.
Against the oracle element by element: planes no longer than a thread's run
(several boundaries in a run), short planes many to a tile (plane
boundaries at and inside runs), planes of about one tile, planes over many
tiles, both directions, inclusive and exclusive, every reduction operator,
integer inputs exactly, reruns bit for bit, neighbours of the output left
alone, and the automatic choice on the shapes it takes."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import assert_close, assert_exact, assert_op_close, bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu
MODES = [(False, False), (False, True), (True, False), (True, True)]
MODE_IDS = ["fwd", "fwd-excl", "rev", "rev-excl"]
SCAN_RUNS = 8    # LIBREDUCE_OPT_SCAN_COLS_VARIANT: narrow planes as segmented class runs
REDUCE_RUNS = 9  # LIBREDUCE_OPT_COLS_VARIANT: the same for reductions
# (outer, N, P): plane lengths L = N*P of 38 to 30003 floats: many planes to
# a 4608-float tile (k >= 2, boundaries inside runs unless L % 36 == 0), one
# plane to a tile, planes over 2 to 7 tiles; plane counts leaving a ragged
# last item; the two bench shapes.
SHAPES = [(100_000, 100, 3), (4096, 4096, 2), (20_001, 19, 2), (30_001, 13, 4), (9000, 767, 3),
          (5000, 2305, 2), (3000, 1537, 3), (2000, 3001, 4), (700, 10_001, 3), (7, 13, 3),
          (3, 333_333, 2), (12_345, 250, 4), (40_000, 9, 4),
          # 5-8 columns (runs of 20, 36, 28 and 24 floats)
          (30_000, 101, 5), (20_001, 5, 5), (3000, 999, 6), (10_000, 7, 6), (7000, 77, 7), (500, 3001, 7),
          (100_000, 100, 8), (9999, 4, 8), (64, 50_001, 5), (3, 200_000, 8),
          # planes no longer than a thread's run: several boundaries in a run
          (500_000, 7, 3), (300_001, 2, 2), (200_000, 5, 4), (100_000, 3, 8), (100_001, 9, 4),
          (70_000, 18, 2), (7, 4, 5), (40_000, 4, 7), (33_333, 12, 3), (50_000, 6, 6),
          # scans of 9, 10, 12 and 14 columns (runs of 36, 20, 36, 28 floats)
          (100_000, 100, 9), (30_001, 37, 10), (20_000, 100, 12), (9999, 101, 14), (200_000, 3, 12),
          (1000, 4001, 9), (64, 10_000, 14), (50_000, 2, 10),
          # scans of 16 and 32 columns (column-group runs of 9 rows, tiles of
          # 288 / 144 rows): many planes to a tile with a ragged last item,
          # planes of 10 rows, planes filling a tile exactly, one plane to a
          # tile, planes over 2 to 70 tiles
          (20_000, 100, 16), (30_001, 13, 16), (9999, 10, 32), (50_001, 11, 32), (10_000, 144, 16),
          (40_000, 72, 32), (5000, 145, 16), (2000, 289, 16), (300, 5001, 32), (64, 10_000, 16),
          (3, 20_000, 16), (7, 12, 16),
          # column groups of other widths: single floats (odd P, runs of 33
          # rows), float2 (P = 2 mod 4, 17 rows) and float4 (9 rows); group
          # counts that do not divide 32 (idle threads past the row groups),
          # 32 groups, tiles starting inside a 16-byte granule, planes of one
          # run and a row, planes over many tiles
          (20_000, 34, 11), (3000, 101, 13), (700, 1001, 15), (5000, 77, 17), (400, 2000, 31),
          (20_000, 18, 18), (4000, 100, 22), (1000, 999, 26), (300, 3001, 30), (2000, 50, 34), (500, 600, 62),
          (20_000, 10, 20), (5000, 100, 24), (1000, 1000, 28), (3000, 99, 36), (1000, 500, 40), (800, 100, 48),
          (500, 300, 64), (100, 2000, 100), (64, 3000, 128), (7, 12, 44),
          # enough planes for items of many planes over several tiles
          (60_000, 40, 20), (80_000, 35, 11), (50_000, 20, 18)]


def scan(x, reverse, exclusive, forced=True, out=None):
    if forced:
        L.set_option(L.OPT_SCAN_COLS_VARIANT, SCAN_RUNS)
    xd = on_device(x)
    y = out if out is not None else on_device(torch.zeros_like(x))
    L.cumsum_f32(xd, 1, reverse=reverse, exclusive=exclusive, out=y)
    L.check()
    return y


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", SHAPES)
def test_scan_against_oracle(shape, reverse, exclusive):
    x = inputs.make(shape, "uniform_pm1", 31)
    y = scan(x, reverse, exclusive)
    ref, scale = oracle.cumsum(x.numpy(), *shape, reverse, exclusive)
    assert_close(y.cpu().numpy(), ref, scale, f"plane runs {shape} rev={reverse} excl={exclusive}")


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", [(40_000, 25, 3), (3000, 2401, 2), (1000, 2500, 4), (200_000, 7, 3), (20_000, 50, 16),
                                   (3000, 1001, 32), (3000, 70, 13), (1000, 300, 22), (500, 200, 40), (50, 700, 128)])
def test_scan_integers_exact_and_bitwise(shape, reverse, exclusive):
    """{0..3} inputs: every prefix is an integer below 2^24, so exact."""
    x = inputs.make(shape, "int:0:3", 32)
    a = scan(x, reverse, exclusive).clone()
    b = scan(x, reverse, exclusive)
    assert bitwise_equal(a, b), "reruns differ"
    ref, _ = oracle.cumsum(x.numpy(), *shape, reverse, exclusive)
    assert_exact(a.cpu().numpy(), ref, f"plane runs integers {shape}")


@pytest.mark.parametrize("op", ["sum", "mean", "max", "min", "norm"])
@pytest.mark.parametrize("shape", [(100_000, 100, 3), (20_001, 19, 2), (9000, 767, 3), (2000, 3001, 4),
                                   (7, 13, 3), (4096, 2305, 2), (40_000, 9, 4), (30_000, 101, 5),
                                   (10_000, 7, 6), (500, 3001, 7), (100_000, 100, 8),
                                   (500_000, 7, 3), (300_001, 2, 2), (100_000, 3, 8), (40_000, 4, 7),
                                   (33_333, 12, 3),
                                   # column groups, 9-128 columns: every group width,
                                   # group counts that do not divide 32, planes of a
                                   # run and a row, one plane over many tiles
                                   (20_000, 34, 9), (5000, 101, 10), (3000, 999, 11), (10_000, 10, 12),
                                   (2000, 77, 13), (700, 2001, 16), (4000, 35, 17), (3000, 100, 20),
                                   (1000, 300, 26), (400, 2000, 31), (2000, 50, 32), (1000, 99, 40),
                                   (300, 1000, 64), (100, 2000, 100), (64, 3000, 128), (7, 12, 44),
                                   (60_000, 40, 20), (80_000, 35, 11), (50_000, 20, 18)])
def test_reduce_against_oracle(shape, op):
    L.set_option(L.OPT_COLS_VARIANT, REDUCE_RUNS)
    x = inputs.make(shape, "uniform_pm1", 33)
    out = L.reduce_axis_op_f32(on_device(x), 1, op)
    L.check()
    o, n, i = shape
    if op == "sum":
        ref, scale = oracle.axis_sum(x.numpy(), o, n, i)
        assert_close(out.cpu().numpy(), ref, scale, f"plane runs sum {shape}")
    else:
        ref, scale = oracle.reduce_op(x.numpy(), o, n, i, op)
        assert_op_close(out, ref, scale, op, n, f"plane runs {op} {shape}")


@pytest.mark.parametrize("op", ["max", "min", "sum"])
@pytest.mark.parametrize("shape", [(5000, 37, 3), (3000, 37, 13)])
def test_reduce_nan_stays_in_its_plane(op, shape):
    """L = 111 (3 columns): plane ends inside runs; 13 columns: column groups."""
    x = inputs.make(shape, "uniform_pm1", 34)
    o, n, i = shape
    x[17, 5, 1] = float("nan")
    x[o - 1, n - 1, 2] = float("nan")
    L.set_option(L.OPT_COLS_VARIANT, REDUCE_RUNS)
    out = L.reduce_axis_op_f32(on_device(x), 1, op).cpu().numpy()
    L.check()
    nan = np.isnan(out.reshape(o, i))
    assert nan[17, 1] and nan[o - 1, 2] and nan.sum() == 2
    if op == "sum":
        ref, scale = oracle.axis_sum(x.numpy(), *shape)
        keep = ~np.isnan(ref)
        assert_close(out[keep], ref[keep], scale[keep], "plane runs sum beside NaN")
    else:
        ref, scale = oracle.reduce_op(x.numpy(), *shape, op)
        assert_op_close(out, ref, scale, op, shape[1], f"plane runs {op} with NaN")


@pytest.mark.parametrize("shape", [(6000, 100, 3), (300, 3001, 4), (100_000, 5, 3), (3000, 99, 11), (500, 1000, 20),
                                   (2000, 40, 34)])
def test_reduce_integers_exact_and_bitwise(shape):
    x = inputs.make(shape, "int:-8:8", 35)
    L.set_option(L.OPT_COLS_VARIANT, REDUCE_RUNS)
    xd = on_device(x)
    a = L.reduce_axis_f32(xd, 1).clone()
    b = L.reduce_axis_f32(xd, 1)
    L.check()
    assert bitwise_equal(a, b)
    ref, _ = oracle.axis_sum(x.numpy(), *shape)
    assert_exact(a.cpu().numpy(), ref, f"plane runs sum integers {shape}")


@pytest.mark.parametrize("reverse", [False, True])
def test_neighbours_untouched(reverse):
    """Output at a 16-byte offset inside a larger buffer of sentinels; planes
    whose boundaries fall inside float4 granules (L = 6002 and L = 38), and
    column-group tiles whose last item ends short of a tile (16 and 32
    columns)."""
    for shape in [(7, 3001, 2), (5001, 19, 2), (1001, 13, 16), (3, 1001, 32), (1001, 35, 11), (13, 37, 18)]:
        x = inputs.make(shape, "uniform01", 36)
        n = x.numel()
        buf = torch.full((n + 12,), 5.0, device="cuda")
        y = buf[4:4 + n].view(shape)
        scan(x, reverse, False, out=y)
        assert torch.all(buf[:4] == 5.0) and torch.all(buf[4 + n:] == 5.0)
        ref, scale = oracle.cumsum(x.numpy(), *shape, reverse, False)
        assert_close(y.cpu().numpy(), ref, scale, f"neighbours {shape}")


@pytest.mark.parametrize("shape,sums", [((100_000, 100, 3), True), ((4096, 4096, 2), True), ((50_000, 40, 4), True),
                                        ((500_000, 7, 3), True), ((100_000, 100, 8), False),
                                        ((100_000, 100, 16), False), ((50_000, 100, 32), False),
                                        ((20_000, 100, 13), False), ((20_000, 100, 22), False),
                                        ((10_000, 100, 40), False)])
def test_automatic_choice_takes_plane_runs(shape, sums):
    """Aligned planes whose items fill the GPU take this form without options:
    the automatic result is the forced one bit for bit (sums of 8 columns keep
    the narrow kernels; sums of 16 and 32 columns have no plane-run form)."""
    x = inputs.make(shape, "uniform_pm1", 37)
    auto = scan(x, False, False, forced=False).clone()
    forced = scan(x, False, False)
    assert bitwise_equal(auto, forced)
    if not sums:
        return
    L.set_option(L.OPT_SCAN_COLS_VARIANT, -1)
    xd = on_device(x)
    auto_sum = L.reduce_axis_f32(xd, 1).clone()
    L.set_option(L.OPT_COLS_VARIANT, REDUCE_RUNS)
    assert bitwise_equal(auto_sum, L.reduce_axis_f32(xd, 1))


def test_misaligned_falls_back():
    """x or y off a 16-byte boundary: another form, still against the oracle."""
    shape = (20_000, 100, 3)
    x = inputs.make(shape, "uniform_pm1", 38)
    L.set_option(L.OPT_SCAN_COLS_VARIANT, SCAN_RUNS)
    xd = on_device(x, 1)
    y = L.cumsum_f32(xd, 1)
    L.check()
    ref, scale = oracle.cumsum(x.numpy(), *shape, False, False)
    assert_close(y.cpu().numpy(), ref, scale, "misaligned plane runs")


# ---- few long planes: the look-back form (one tile per block) ----------------------

SCAN_LOOKBACK = 9  # LIBREDUCE_OPT_SCAN_COLS_VARIANT: the same tiles, a plane over blocks
# One plane of ~650 tiles (two levels of the 32-ary tree), planes of 7, 3 and
# one tile, plane lengths that are and are not multiples of the 16-byte
# granule (and of 12 floats for 3 columns), a plane of 33 tiles (a level-1
# parent completed by its 32nd tile).
LB_SHAPES = [(1, 1_000_003, 3), (3, 400_000, 4), (5, 250_001, 2), (7, 10_001, 3), (4, 4609, 2),
             (3, 50, 3), (2, 38_017, 4), (1, 76_033, 2),
             (1, 300_001, 5), (2, 100_003, 6), (3, 90_001, 7), (1, 500_000, 8), (5, 2000, 7)]


def scan_lb(x, reverse, exclusive, forced=True):
    if forced:
        L.set_option(L.OPT_SCAN_COLS_VARIANT, SCAN_LOOKBACK)
    y = L.cumsum_f32(on_device(x), 1, reverse=reverse, exclusive=exclusive)
    L.check()
    return y


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", LB_SHAPES)
def test_lookback_against_oracle(shape, reverse, exclusive):
    x = inputs.make(shape, "uniform_pm1", 41)
    y = scan_lb(x, reverse, exclusive)
    ref, scale = oracle.cumsum(x.numpy(), *shape, reverse, exclusive)
    assert_close(y.cpu().numpy(), ref, scale, f"plane look-back {shape} rev={reverse} excl={exclusive}")


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_lookback_integers_exact_and_bitwise(reverse, exclusive):
    """{0..3}: every prefix below 2^24 (at most 3 * 1.3e6), so exact."""
    shape = (2, 1_300_001, 2)
    x = inputs.make(shape, "int:0:3", 42)
    a = scan_lb(x, reverse, exclusive).clone()
    b = scan_lb(x, reverse, exclusive)
    assert bitwise_equal(a, b), "reruns differ"
    ref, _ = oracle.cumsum(x.numpy(), *shape, reverse, exclusive)
    assert_exact(a.cpu().numpy(), ref, "plane look-back integers")


@pytest.mark.parametrize("lag", [64, 640, 4096])
def test_lookback_lags(lag):
    """Any lag gives the same bits (the carries never depend on timing)."""
    shape = (1, 3_000_001, 3)
    x = inputs.make(shape, "uniform_pm1", 43)
    base = scan_lb(x, False, False).clone()
    L.set_option(L.OPT_LOOKBACK_LAG, lag)
    assert bitwise_equal(base, scan_lb(x, False, False))


def test_lookback_is_the_automatic_choice_for_few_long_planes():
    shape = (1, 40_000_000, 4)
    x = inputs.make(shape, "uniform_pm1", 44)
    auto = scan_lb(x, False, False, forced=False).clone()
    assert bitwise_equal(auto, scan_lb(x, False, False))


def test_lookback_bounded_wait_reports_timeout():
    """A tile that never publishes (chosen on the host) makes the waits
    behind it run out: the host reads TIMEOUT, and the next call is right."""
    shape = (1, 2_000_000, 3)
    x = inputs.make(shape, "uniform01", 45)
    xd = on_device(x)
    L.set_option(L.OPT_SCAN_COLS_VARIANT, SCAN_LOOKBACK)
    L.set_option(L.OPT_SPIN_LIMIT, 2000)
    L.set_option(L.OPT_STALL_TILE, 5)
    L.cumsum_f32(xd, 1)
    with pytest.raises(L.LibreduceError) as ei:
        L.check()
    assert ei.value.status == L.ERR_TIMEOUT
    L.set_option(L.OPT_STALL_TILE, -1)
    L.set_option(L.OPT_SPIN_LIMIT, 0)
    L.check()
    ref, scale = oracle.cumsum(x.numpy(), *shape, False, False)
    assert_close(L.cumsum_f32(xd, 1).cpu().numpy(), ref, scale, "after timeout")


# ---- few long planes as column groups (6-128 columns): k_planes_cg_lb ----------
# Every group width (float for odd widths, float2, float4), group counts that do
# not divide 32, 32 groups, tiles starting inside a 16-byte granule, planes of
# two tiles, of 33 tiles (a level-1 parent completed by its 32nd tile) and of
# ~1700 tiles (two levels and a third); the existing shapes of 6-8 columns
# above take it too.
CG_LB_SHAPES = [(1, 500_003, 11), (3, 200_000, 16), (5, 100_001, 13), (2, 60_000, 31), (4, 30_000, 40),
                (7, 1300, 20), (1, 300_000, 6), (2, 100_000, 18), (1, 2_000_000, 10), (3, 9801, 22),
                (2, 20_000, 128), (1, 5000, 64)]


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", CG_LB_SHAPES)
def test_column_group_lookback_against_oracle(shape, reverse, exclusive):
    x = inputs.make(shape, "uniform_pm1", 46)
    y = scan_lb(x, reverse, exclusive)
    ref, scale = oracle.cumsum(x.numpy(), *shape, reverse, exclusive)
    assert_close(y.cpu().numpy(), ref, scale, f"column-group look-back {shape} rev={reverse} excl={exclusive}")


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", [(2, 400_001, 13), (1, 300_000, 20)])
def test_column_group_lookback_integers_exact_and_bitwise(shape, reverse, exclusive):
    """{0..3}: every prefix below 2^24, so exact."""
    x = inputs.make(shape, "int:0:3", 47)
    a = scan_lb(x, reverse, exclusive).clone()
    b = scan_lb(x, reverse, exclusive)
    assert bitwise_equal(a, b), "reruns differ"
    ref, _ = oracle.cumsum(x.numpy(), *shape, reverse, exclusive)
    assert_exact(a.cpu().numpy(), ref, f"column-group look-back integers {shape}")


@pytest.mark.parametrize("lag", [64, 640, 4096])
def test_column_group_lookback_lags(lag):
    shape = (1, 1_000_001, 16)
    x = inputs.make(shape, "uniform_pm1", 48)
    base = scan_lb(x, True, False).clone()
    L.set_option(L.OPT_LOOKBACK_LAG, lag)
    assert bitwise_equal(base, scan_lb(x, True, False))


@pytest.mark.parametrize("shape", [(1, 2_000_000, 16), (8, 200_000, 13), (3, 300_000, 24)])
def test_column_group_lookback_is_the_automatic_choice(shape):
    x = inputs.make(shape, "uniform_pm1", 49)
    auto = scan_lb(x, False, False, forced=False).clone()
    assert bitwise_equal(auto, scan_lb(x, False, False))


def test_column_group_lookback_bounded_wait_reports_timeout():
    shape = (1, 500_000, 16)
    x = inputs.make(shape, "uniform01", 50)
    xd = on_device(x)
    L.set_option(L.OPT_SCAN_COLS_VARIANT, SCAN_LOOKBACK)
    L.set_option(L.OPT_SPIN_LIMIT, 2000)
    L.set_option(L.OPT_STALL_TILE, 5)
    L.cumsum_f32(xd, 1)
    with pytest.raises(L.LibreduceError) as ei:
        L.check()
    assert ei.value.status == L.ERR_TIMEOUT
    L.set_option(L.OPT_STALL_TILE, -1)
    L.set_option(L.OPT_SPIN_LIMIT, 0)
    L.check()
    ref, scale = oracle.cumsum(x.numpy(), *shape, False, False)
    assert_close(L.cumsum_f32(xd, 1).cpu().numpy(), ref, scale, "after timeout")
