"""Scans of narrow planes of 2 or 4 columns read flat (GPU): [outer, N, inner]
along N with inner in {2, 4} is scanned by the row kernels over each plane's
N*inner floats, element e in column class e % inner (float4 tiles one block
per plane, or the L2 look-back for few planes).  Against the oracle element
by element: both directions, inclusive and exclusive, planes of whole and
partial float4s, x and y at every shared 4-byte offset, both forms forced,
integer inputs exactly, reruns bit for bit, and a host-chosen stall that
makes the look-back's waits run out."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import assert_close, assert_exact, bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu
MODES = [(False, False), (False, True), (True, False), (True, True)]
MODE_IDS = ["fwd", "fwd-excl", "rev", "rev-excl"]
PERIOD_ROWS = 7  # LIBREDUCE_OPT_SCAN_COLS_VARIANT: planes of 2 or 4 columns as flat rows
# Many planes (one block per plane), few planes (look-back), plane lengths in
# floats that are and are not multiples of 4, single-tile and many-tile planes.
SHAPES = [(4096, 4096, 2), (300, 5000, 4), (513, 2049, 2), (33, 3001, 4), (1, 4_000_000, 4),
          (2, 3_000_001, 2), (1, 1_234_567, 2), (3, 777_777, 4), (5, 1025, 2), (1, 6000, 4)]


def scan(x, reverse, exclusive, offset=0, forced=True, strategy=0):
    if forced:
        L.set_option(L.OPT_SCAN_COLS_VARIANT, PERIOD_ROWS)
    L.set_option(L.OPT_SCAN_STRATEGY, strategy)
    xd = on_device(x, offset)
    y = on_device(torch.zeros_like(x), offset)
    L.cumsum_f32(xd, 1, reverse=reverse, exclusive=exclusive, out=y)
    L.check()
    return y


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", SHAPES)
def test_against_oracle(shape, reverse, exclusive):
    x = inputs.make(shape, "uniform_pm1", 21)
    y = scan(x, reverse, exclusive)
    ref, scale = oracle.cumsum(x.numpy(), *shape, reverse, exclusive)
    assert_close(y.cpu().numpy(), ref, scale, f"period planes {shape} rev={reverse} excl={exclusive}")


@pytest.mark.parametrize("offset", [1, 2, 3])
@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_offsets(offset, reverse, exclusive):
    for shape in [(100, 5001, 2), (1, 2_000_003, 4)]:
        x = inputs.make(shape, "uniform01", 22)
        y = scan(x, reverse, exclusive, offset)
        ref, scale = oracle.cumsum(x.numpy(), *shape, reverse, exclusive)
        assert_close(y.cpu().numpy(), ref, scale, f"period planes {shape} at +{offset}")


@pytest.mark.parametrize("strategy", [1, 2])
@pytest.mark.parametrize("inner", [2, 4])
def test_both_forms_integers_exact_and_bitwise(strategy, inner):
    shape = (3, 1_000_000 // inner + 7, inner)
    x = inputs.make(shape, "int:0:3", 23)
    ref, _ = oracle.cumsum(x.numpy(), *shape, False, False)
    a = scan(x, False, False, strategy=strategy).clone()
    b = scan(x, False, False, strategy=strategy)
    assert bitwise_equal(a, b)
    # Suffix/prefix sums here stay below 2^24 (at most 3 * 1e6 / inner).
    assert_exact(a.cpu().numpy(), ref, f"period planes integers strategy {strategy}")


def test_automatic_choice_matches_forced():
    """Without options, 2-column planes of at least 4096 floats take this path."""
    x = inputs.make((64, 4096, 2), "uniform01", 24)
    auto = scan(x, True, False, forced=False)
    forced = scan(x, True, False)
    assert bitwise_equal(auto, forced)


def test_neighbours_untouched():
    shape = (7, 3001, 2)  # plane of 6002 floats: partial float4s at both ends
    x = inputs.make(shape, "uniform01", 25)
    n = x.numel()
    L.set_option(L.OPT_SCAN_COLS_VARIANT, PERIOD_ROWS)
    xd = on_device(x, 1)
    buf = torch.full((n + 8,), 5.0, device="cuda")
    y = buf[1:1 + n].view(shape)
    L.cumsum_f32(xd, 1, out=y)
    L.check()
    assert buf[0].item() == 5.0 and torch.all(buf[1 + n:] == 5.0)
    ref, scale = oracle.cumsum(x.numpy(), *shape, False, False)
    assert_close(y.cpu().numpy(), ref, scale, "neighbours")


@pytest.mark.parametrize("inner", [2, 4])
def test_bounded_wait_reports_timeout(inner):
    """A tile that never publishes (chosen on the host) makes the look-back's
    waits behind it run out: the host reads TIMEOUT and the library keeps
    working."""
    shape = (1, 600_000 // inner * 4, inner)
    x = inputs.make(shape, "uniform01", 26)
    L.set_option(L.OPT_SCAN_COLS_VARIANT, PERIOD_ROWS)
    L.set_option(L.OPT_SCAN_STRATEGY, 2)
    L.set_option(L.OPT_SPIN_LIMIT, 2000)
    L.set_option(L.OPT_STALL_TILE, 5)
    xd = on_device(x)
    L.cumsum_f32(xd, 1, reverse=True)
    with pytest.raises(L.LibreduceError) as ei:
        L.check()
    assert ei.value.status == L.ERR_TIMEOUT
    L.set_option(L.OPT_STALL_TILE, -1)
    L.set_option(L.OPT_SPIN_LIMIT, 0)
    L.check()
    ref, scale = oracle.cumsum(x.numpy(), *shape, True, False)
    assert_close(L.cumsum_f32(xd, 1, reverse=True).cpu().numpy(), ref, scale, "after timeout")
