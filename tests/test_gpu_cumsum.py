"""cumsum_f32 (forward / reverse, inclusive / exclusive, any axis) against the
oracle (GPU)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import assert_close, assert_exact, bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
MODES = [(False, False), (False, True), (True, False), (True, True)]
MODE_IDS = ["fwd", "fwd-excl", "rev", "rev-excl"]


def run(x_cpu, dim, reverse, exclusive, offset=0, out_offset=0):
    xd = on_device(x_cpu, offset)
    y = on_device(torch.zeros_like(x_cpu), out_offset)
    L.cumsum_f32(xd, dim, reverse=reverse, exclusive=exclusive, out=y)
    L.check()
    return y.cpu().numpy()


def check(shape, dim, reverse, exclusive, dist="uniform_pm1", seed=4, offset=0, out_offset=0):
    x = inputs.make(shape, dist, seed)
    o, n, i = L.canonical_axis(x.shape, dim)
    ref, scale = oracle.cumsum(x.numpy(), o, n, i, reverse, exclusive)
    got = run(x, dim, reverse, exclusive, offset, out_offset)
    assert_close(got.reshape(-1), ref.reshape(-1), scale.reshape(-1),
                 f"cumsum {shape} dim={dim} rev={reverse} excl={exclusive} off={offset}/{out_offset}")
    return got, ref


def test_worked_examples():
    with open(os.path.join(GOLDEN, "exclusive_scan_worked_example.json")) as f:
        cases = json.load(f)["cases"]
    with open(os.path.join(GOLDEN, "rcumsum_worked_examples.json")) as f:
        cases += [dict(c, reverse=True, exclusive=False) for c in json.load(f)["cases"]]
    for c in cases:
        x = torch.tensor([c["x"]], dtype=torch.float32)
        got = run(x, 1, c["reverse"], c["exclusive"])
        assert got.reshape(-1).tolist() == [float(v) for v in c["y"]], c


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("rows,n", [(1, 1), (3, 5), (2, 4096), (5, 8193), (37, 32768), (300, 1001),
                                    (1, 1_000_003), (3, 200_004)])
def test_rows(rows, n, reverse, exclusive):
    got, ref = check((rows, n), 1, reverse, exclusive)
    if exclusive:
        edge = 0 if not reverse else n - 1
        assert np.all(got[:, edge] == 0.0)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("strategy", [1, 2, 3, 4])
def test_rows_every_strategy(strategy, reverse, exclusive):
    L.set_option(L.OPT_SCAN_STRATEGY, strategy)
    check((3, 100_000), 1, reverse, exclusive)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("offset,out_offset", [(1, 0), (2, 3)])
def test_rows_misaligned(offset, out_offset, reverse, exclusive):
    check((4, 50_001), 1, reverse, exclusive, offset=offset, out_offset=out_offset)
    for strategy in (2, 4):
        L.set_option(L.OPT_SCAN_STRATEGY, strategy)
        check((1, 300_000), 1, reverse, exclusive, offset=offset, out_offset=out_offset)


# Rows of any length and any 4-byte offset (shared by x and y) run on the
# float4 paths as aligned "virtual rows": the float4 items at a row's two
# edges are masked.  N = 3 * 8192 - 1 over 4 rows gives rows whose virtual
# lengths differ by one float4 across a tile boundary, so some rows end
# with a tile that holds none of their elements.
VIRTUAL_ROWS = [(4, 3 * 8192 - 1), (5, 8192 + 2), (3, 100_003), (2, 32767), (9, 4097), (1, 5), (6, 3)]


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("strategy", [1, 2, 3, 4])
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_rows_virtual_float4(strategy, offset, reverse, exclusive):
    L.set_option(L.OPT_SCAN_STRATEGY, strategy)
    for rows, n in VIRTUAL_ROWS:
        got, _ = check((rows, n), 1, reverse, exclusive, offset=offset, out_offset=offset)
        if exclusive:
            assert np.all(got[:, n - 1 if reverse else 0] == 0.0)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("strategy", [1, 2, 3, 4])
def test_rows_virtual_integers_exact(strategy, reverse, exclusive):
    """Small integers sum exactly, so a masked edge item that leaked into a
    tile total (or a dropped element) changes some output bit."""
    L.set_option(L.OPT_SCAN_STRATEGY, strategy)
    for rows, n in [(4, 3 * 8192 - 1), (3, 20_001)]:
        for offset in (1, 3):
            x = inputs.make((rows, n), "int:0:3", 17 + offset)
            ref, _ = oracle.cumsum(x.numpy(), rows, n, 1, reverse, exclusive)
            got = run(x, 1, reverse, exclusive, offset, offset)
            assert_exact(got.reshape(-1), ref.reshape(-1), f"[{rows},{n}] s={strategy} off={offset}")


def test_rows_virtual_neighbours_untouched():
    """Stores at a row's edges write only the row's own elements: the floats
    around a misaligned output keep their values."""
    for strategy in (1, 2, 3, 4):
        L.set_option(L.OPT_SCAN_STRATEGY, strategy)
        for reverse in (False, True):
            x = inputs.make((3, 8192 + 2), "uniform01", 5)
            n = x.numel()
            buf = torch.full((n + 8,), 7.0, device="cuda")
            y = buf[1:1 + n].view(x.shape)
            L.cumsum_f32(on_device(x, 1), 1, reverse=reverse, out=y)
            L.check()
            rest = torch.cat([buf[:1], buf[1 + n:]]).cpu()
            assert torch.all(rest == 7.0), (strategy, reverse)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape,dim", [((4, 9, 7), 1), ((2, 1000, 64), 1), ((3, 257, 33), 1),
                                       ((1, 5000, 4096), 1), ((600, 8), 0), ((7, 6, 5, 4), 2),
                                       ((16, 4096, 4095), 1)])
def test_axis(shape, dim, reverse, exclusive):
    check(shape, dim, reverse, exclusive)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_axis_misaligned_and_long(reverse, exclusive):
    check((2, 700, 36), 1, reverse, exclusive, offset=1)
    check((2, 300_000, 4), 1, reverse, exclusive)  # long axis: blocked running sum


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_integer_inputs_exact(reverse, exclusive):
    for shape, dim in (((64, 32768), 1), ((3, 4000, 36), 1), ((1, 1 << 20), 1)):
        x = inputs.make(shape, "int:0:3", 3)
        o, n, i = L.canonical_axis(x.shape, dim)
        ref, _ = oracle.cumsum(x.numpy(), o, n, i, reverse, exclusive)
        assert_exact(run(x, dim, reverse, exclusive).reshape(-1), ref.reshape(-1), f"int {shape}")


def test_deterministic_bitwise():
    for shape, dim in (((1, 1 << 24), 1), ((128, 4096, 63), 1), ((512, 32768), 1)):
        xd = on_device(inputs.make(shape, "uniform01", 5))
        for reverse, exclusive in MODES:
            outs = [L.cumsum_f32(xd, dim, reverse=reverse, exclusive=exclusive).clone() for _ in range(3)]
            L.check()
            for o in outs[1:]:
                assert bitwise_equal(outs[0], o), (shape, reverse, exclusive)


def test_reverse_entry_point_matches():
    xd = on_device(inputs.make((5, 70_000), "uniform01", 6))
    a = L.reverse_cumsum_f32(xd)
    b = L.cumsum_f32(xd, 1, reverse=True)
    L.check()
    assert bitwise_equal(a, b)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape,segs,offset", [((3, 1000, 36), 7, 0), ((2, 777, 4096), 3, 0),
                                               ((4, 301, 33), 5, 0), ((1, 5000, 4096), 64, 1),
                                               ((2, 130, 12), 130, 0), ((2, 100, 8), 1000, 0),
                                               ((1, 70_001, 4), 0, 0), ((2, 3000, 5), 0, 2)])
def test_axis_segmented(shape, segs, offset, reverse, exclusive):
    """The column scan cut into segments: segment sums, a scan of the sums,
    then every segment rescanned from its carry.  segs > 0 forces the count
    (clamped to one row per segment); 0 leaves it to the library, which cuts
    the axis when there are too few columns to fill the GPU."""
    if segs:
        L.set_option(L.OPT_AXIS_SPLIT, segs)
    got, _ = check(shape, 1, reverse, exclusive, offset=offset)
    if exclusive:
        edge = 0 if not reverse else shape[1] - 1
        assert np.all(got[:, edge, :] == 0.0)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_axis_segmented_integers_exact(reverse, exclusive):
    for shape, segs in (((3, 4000, 36), 9), ((2, 2048, 7), 64), ((1, 100_000, 8), 0)):
        L.set_option(L.OPT_AXIS_SPLIT, segs)
        x = inputs.make(shape, "int:0:3", 8)
        o, n, i = L.canonical_axis(x.shape, 1)
        ref, _ = oracle.cumsum(x.numpy(), o, n, i, reverse, exclusive)
        assert_exact(run(x, 1, reverse, exclusive).reshape(-1), ref.reshape(-1), f"int {shape} segs={segs}")


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_axis_every_block_shape(variant, reverse, exclusive):
    """Each column-scan block shape (scalar 2x4 warps, float4 2x4, float4 1x8),
    on shapes with ragged column tiles and ragged row tiles, rows of every
    16-byte misalignment, single pass and segmented; float4 shapes fall back
    to the automatic choice where rows are not aligned."""
    L.set_option(L.OPT_SCAN_COLS_VARIANT, variant)
    for shape, segs, off in (((3, 1001, 388), 0, 0), ((2, 333, 132), 5, 0), ((5, 77, 4096), 0, 0),
                             ((2, 900, 36), 3, 0), ((2, 130, 37), 0, 0), ((3, 500, 4095), 0, 0),
                             ((2, 300, 258), 4, 1), ((2, 97, 301), 0, 3), ((4, 64, 1000), 0, 2)):
        L.set_option(L.OPT_AXIS_SPLIT, segs)
        check(shape, 1, reverse, exclusive, offset=off, out_offset=(off * 3) % 4)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape,segs,offset", [((2, 30000, 4), 0, 0), ((5, 777, 3), 0, 0), ((3, 1000, 32), 0, 0),
                                               ((2, 5000, 128), 0, 0), ((4, 1001, 12), 3, 0),
                                               ((1, 200000, 2), 0, 0), ((100, 300, 7), 0, 0),
                                               ((2, 70001, 16), 17, 0), ((3, 5000, 8), 0, 1),
                                               ((2, 3001, 20), 5, 2), ((1, 3, 5), 0, 0), ((2, 1, 4), 0, 0),
                                               ((3, 4097, 31), 0, 3), ((1, 100000, 33), 0, 0),
                                               ((3, 2000, 100), 0, 0), ((2, 3000, 255), 4, 0),
                                               ((4, 1000, 256), 0, 1), ((600, 50, 64), 0, 0)])
@pytest.mark.parametrize("form", [-1, 3, 4], ids=["auto", "block", "warp"])
def test_axis_narrow(shape, segs, offset, reverse, exclusive, form):
    """Rows of at most 32 column groups: the narrow scan, with tiles staged in
    shared memory (block form) or a warp per (plane, segment) scanning row
    groups with shuffles (warp form), one unit per plane or cut into segments
    (forced, or automatic when outer is small)."""
    L.set_option(L.OPT_SCAN_COLS_VARIANT, form)
    if segs:
        L.set_option(L.OPT_AXIS_SPLIT, segs)
    got, _ = check(shape, 1, reverse, exclusive, offset=offset, out_offset=(offset * 3) % 4)
    if exclusive:
        edge = 0 if not reverse else shape[1] - 1
        assert np.all(got[:, edge, :] == 0.0)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("form", [3, 4], ids=["block", "warp"])
def test_axis_narrow_integers_exact(reverse, exclusive, form):
    L.set_option(L.OPT_SCAN_COLS_VARIANT, form)
    for shape, segs in (((3, 4000, 4), 0), ((2, 20001, 3), 9), ((1, 100_000, 16), 0), ((4, 999, 32), 5),
                        ((5000, 7, 3), 0)):
        L.set_option(L.OPT_AXIS_SPLIT, segs)
        x = inputs.make(shape, "int:0:3", 8)
        o, n, i = L.canonical_axis(x.shape, 1)
        ref, _ = oracle.cumsum(x.numpy(), o, n, i, reverse, exclusive)
        assert_exact(run(x, 1, reverse, exclusive).reshape(-1), ref.reshape(-1), f"narrow int {shape} segs={segs}")


def test_axis_narrow_wide_forced_agree():
    """The wide column scan forced on narrow rows also matches the oracle."""
    L.set_option(L.OPT_SCAN_COLS_VARIANT, 0)
    for shape in ((2, 3000, 4), (3, 1000, 7), (2, 500, 32)):
        check(shape, 1, True, False)
        check(shape, 1, False, True)


# The single-pass column look-back (OPT_SCAN_COLS_VARIANT 5): 256-row x
# 32-column tiles, tickets column tile fastest, a 32-ary look-back per column.
COL_LB = 5


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape,offset", [((2, 1000, 64), 0), ((3, 257, 33), 1), ((1, 9000, 40), 2),
                                          ((2, 600, 4095), 3), ((1, 256, 32), 0), ((4, 255, 5), 0),
                                          ((1, 1, 70), 0), ((2, 20, 3), 1), ((1, 270_000, 3), 0)])
def test_axis_lookback(shape, offset, reverse, exclusive):
    """Several tiles per unit, ragged row and column tiles, fewer rows than a
    tile, one to three look-back levels (9000 rows: 36 tiles, two levels;
    270000 rows: 1055 tiles, three), any 4-byte offset of x and of y."""
    L.set_option(L.OPT_SCAN_COLS_VARIANT, COL_LB)
    got, _ = check(shape, 1, reverse, exclusive, offset=offset, out_offset=(offset + 1) % 4)
    if exclusive:
        assert np.all(got[:, shape[1] - 1 if reverse else 0, :] == 0.0)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_axis_lookback_integers_exact(reverse, exclusive):
    L.set_option(L.OPT_SCAN_COLS_VARIANT, COL_LB)
    for shape in ((2, 9000, 40), (1, 2000, 4095), (3, 300, 7)):
        x = inputs.make(shape, "int:0:3", 9)
        o, n, i = L.canonical_axis(x.shape, 1)
        ref, _ = oracle.cumsum(x.numpy(), o, n, i, reverse, exclusive)
        assert_exact(run(x, 1, reverse, exclusive).reshape(-1), ref.reshape(-1), f"look-back int {shape}")


def test_axis_lookback_bitwise_any_lag():
    """Every sum runs in a fixed order, so the result does not depend on the
    lag between a tile's two touches (which changes the timing and which
    waits happen) and is bit-identical across runs."""
    L.set_option(L.OPT_SCAN_COLS_VARIANT, COL_LB)
    x = on_device(inputs.make((2, 9000, 100), "normal", 12))
    first = L.cumsum_f32(x, 1, reverse=True)
    for lag in (0, 1, 7, 64, 5000, 0):
        L.set_option(L.OPT_LOOKBACK_LAG, lag)
        assert bitwise_equal(L.cumsum_f32(x, 1, reverse=True), first), lag
    L.check()


def test_axis_lookback_bounded_wait_reports_timeout():
    """A tile that never publishes (chosen on the host) makes the waits behind
    it run out: the kernel returns, the host reads TIMEOUT, and the library
    keeps working afterwards."""
    L.set_option(L.OPT_SCAN_COLS_VARIANT, COL_LB)
    x = on_device(inputs.make((1, 4096, 64), "uniform01", 3))
    L.set_option(L.OPT_SPIN_LIMIT, 2000)
    L.set_option(L.OPT_STALL_TILE, 3)
    L.cumsum_f32(x, 1)
    with pytest.raises(L.LibreduceError) as ei:
        L.check()
    assert ei.value.status == L.ERR_TIMEOUT
    L.set_option(L.OPT_STALL_TILE, -1)
    L.set_option(L.OPT_SPIN_LIMIT, 0)
    L.check()  # the error word was cleared
    xc = x.cpu()
    ref, scale = oracle.cumsum(xc.numpy(), 1, 4096, 64, False, False)
    assert_close(L.cumsum_f32(x, 1).cpu().numpy().reshape(-1), ref.reshape(-1), scale.reshape(-1), "after timeout")


def test_axis_lookback_is_the_automatic_choice_for_few_units():
    """[1, 5000, 4096] has 16 column tiles of the wide kernel: the library
    takes the one-launch look-back instead of the three-pass segmented scan,
    and both match the oracle."""
    x = inputs.make((1, 5000, 4096), "uniform_pm1", 5)
    ref, scale = oracle.cumsum(x.numpy(), 1, 5000, 4096, True, False)
    xd = on_device(x)
    n0 = L.launch_count()
    auto = L.cumsum_f32(xd, 1, reverse=True)
    L.check()
    assert L.launch_count() - n0 == 1
    assert_close(auto.cpu().numpy().reshape(-1), ref.reshape(-1), scale.reshape(-1), "automatic")
    L.set_option(L.OPT_AXIS_SPLIT, 8)  # a forced split keeps the three-pass form
    n0 = L.launch_count()
    three = L.cumsum_f32(xd, 1, reverse=True)
    L.check()
    assert L.launch_count() - n0 == 3
    assert_close(three.cpu().numpy().reshape(-1), ref.reshape(-1), scale.reshape(-1), "three passes")


def test_axis_lookback_caller_workspace_matches():
    x = on_device(inputs.make((2, 3000, 300), "normal", 6))
    L.set_option(L.OPT_SCAN_COLS_VARIANT, COL_LB)
    plain = L.cumsum_f32(x, 1, exclusive=True)
    ws = L.workspace(L.cumsum_ws_f32(x, 1, exclusive=True))
    got = L.cumsum_ws_f32(x, 1, exclusive=True, ws=ws)
    L.check_ws(ws)
    assert bitwise_equal(got, plain)


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_narrow_few_planes_take_the_lookback(reverse, exclusive):
    """Few planes of narrow float4 rows whose columns fill 32-column tiles are
    scanned by the single-pass column look-back (one launch) instead of the
    three-pass segmented narrow scan; both agree with the oracle."""
    for shape in ((1, 200_000, 32), (2, 60_000, 96)):
        x = inputs.make(shape, "uniform_pm1", 21)
        o, n, i = L.canonical_axis(x.shape, 1)
        ref, scale = oracle.cumsum(x.numpy(), o, n, i, reverse, exclusive)
        xd = on_device(x)
        n0 = L.launch_count()
        got = L.cumsum_f32(xd, 1, reverse=reverse, exclusive=exclusive)
        L.check()
        assert L.launch_count() - n0 == 1, shape
        assert_close(got.cpu().numpy().reshape(-1), ref.reshape(-1), scale.reshape(-1), f"look-back {shape}")
        L.set_option(L.OPT_SCAN_COLS_VARIANT, 3)  # the narrow kernel, segmented
        n0 = L.launch_count()
        three = L.cumsum_f32(xd, 1, reverse=reverse, exclusive=exclusive)
        L.check()
        assert L.launch_count() - n0 == 3, shape
        assert_close(three.cpu().numpy().reshape(-1), ref.reshape(-1), scale.reshape(-1), f"narrow {shape}")
        L.set_option(L.OPT_SCAN_COLS_VARIANT, -1)


# Many short rows (N <= 2048): chunks of whole rows staged in shared memory,
# each row scanned by a group of 1..32 lanes (OPT_SCAN_STRATEGY 5 forces it;
# the automatic choice for such rows).
SHORT_N = [1, 2, 3, 5, 6, 8, 16, 31, 32, 33, 40, 50, 64, 65, 99, 100, 127, 130, 255, 256, 257, 258, 1000, 1002,
           1024, 2046, 2047, 2048]


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("strategy", [0, 5])
def test_short_rows(strategy, reverse, exclusive):
    """Every lane-group size and its boundaries; row counts that leave a
    partial last chunk; 16-byte loads (aligned, N % 4 == 0) and 4-byte loads
    (N % 4 != 0, or x and y at an odd offset); rows unpadded in shared memory
    (one lane per row, N odd)."""
    L.set_option(L.OPT_SCAN_STRATEGY, strategy)
    for n in SHORT_N:
        rows = 3 * max(1, 6144 // n) + 7
        for offset in (0, 1):
            got, _ = check((rows, n), 1, reverse, exclusive, offset=offset, out_offset=offset)
            if exclusive:
                assert np.all(got[:, n - 1 if reverse else 0] == 0.0), n


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_short_rows_integers_exact(reverse, exclusive):
    for n in (7, 32, 66, 100, 1024):
        x = inputs.make((5000, n), "int:0:3", 31)
        ref, _ = oracle.cumsum(x.numpy(), 5000, n, 1, reverse, exclusive)
        assert_exact(run(x, 1, reverse, exclusive).reshape(-1), ref.reshape(-1), f"short rows int N={n}")


def test_short_rows_deterministic_bitwise():
    x = on_device(inputs.make((100_000, 100), "normal", 33))
    first = L.cumsum_f32(x, 1, reverse=True)
    for _ in range(3):
        assert bitwise_equal(L.cumsum_f32(x, 1, reverse=True), first)
    L.check()
