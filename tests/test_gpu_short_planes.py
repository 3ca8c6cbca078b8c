"""Narrow planes by the short-row kernels (GPU): [outer, N, inner] scanned or
reduced along N with N <= 2048, chunks of whole planes staged transposed so
every column is a row.  Against the oracle element by element, over plane
shapes that give every lane plan (one lane per column, groups of 4 to 32
lanes, runs kept in registers or walked in place), 16-byte and 4-byte loads,
pointers at every 4-byte offset, chunks with a ragged last plane count, the
integer inputs exactly and reruns bit for bit."""
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
# (outer, N, inner): N from 1 to 2048 (one lane per column up to 64 / 159,
# lane groups beyond), inner from 2 to 256, plane sizes with and without
# whole float4s, plane counts that leave a ragged last chunk.
SHAPES = [(100_000, 100, 3), (4097, 5, 2), (3001, 64, 4), (999, 159, 3), (1000, 160, 2), (513, 33, 7),
          (257, 1024, 2), (37, 2048, 1 + 1), (65, 200, 12), (129, 11, 256), (7, 1, 5), (2000, 3, 33)]


def scan_check(shape, reverse, exclusive, offset=0, out_offset=0, dist="uniform_pm1", forced=False):
    x = inputs.make(shape, dist, 5)
    if forced:
        L.set_option(L.OPT_SCAN_COLS_VARIANT, 6)
    xd = on_device(x, offset)
    y = on_device(torch.zeros_like(x), out_offset)
    L.cumsum_f32(xd, 1, reverse=reverse, exclusive=exclusive, out=y)
    L.check()
    o, n, i = shape
    ref, scale = oracle.cumsum(x.numpy(), o, n, i, reverse, exclusive)
    return y, ref, scale


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape", SHAPES)
def test_scan(shape, reverse, exclusive):
    # Forced: some of these shapes take the plane-run kernel by default.
    y, ref, scale = scan_check(shape, reverse, exclusive, forced=True)
    assert_close(y.cpu().numpy(), ref, scale, f"planes scan {shape} rev={reverse} excl={exclusive}")


@pytest.mark.parametrize("offset,out_offset", [(1, 1), (2, 3), (3, 0)])
@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_scan_misaligned(offset, out_offset, reverse, exclusive):
    for shape in [(5000, 100, 4), (3000, 37, 3)]:
        y, ref, scale = scan_check(shape, reverse, exclusive, offset, out_offset)
        assert_close(y.cpu().numpy(), ref, scale, f"planes scan {shape} at +{offset}/+{out_offset}")


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_scan_forced_large_planes(reverse, exclusive):
    """Planes beyond the prefetched chunk (up to the shared memory), forced."""
    for shape in [(300, 2048, 2), (100, 1500, 4), (61, 700, 8)]:
        y, ref, scale = scan_check(shape, reverse, exclusive, forced=True)
        assert_close(y.cpu().numpy(), ref, scale, f"forced planes scan {shape}")


@pytest.mark.parametrize("reverse,exclusive", MODES, ids=MODE_IDS)
def test_scan_integers_exact_and_bitwise(reverse, exclusive):
    shape = (20_000, 100, 3)
    x = inputs.make(shape, "int:0:3", 6)
    xd = on_device(x)
    a = L.cumsum_f32(xd, 1, reverse=reverse, exclusive=exclusive).clone()
    b = L.cumsum_f32(xd, 1, reverse=reverse, exclusive=exclusive)
    L.check()
    assert bitwise_equal(a, b)
    ref, _ = oracle.cumsum(x.numpy(), *shape, reverse, exclusive)
    assert_exact(a.cpu().numpy(), ref, "planes scan integers")


def test_scan_neighbours_untouched():
    """Outputs at a 4-byte offset: the floats around y keep their values."""
    shape = (3000, 50, 3)
    x = inputs.make(shape, "uniform01", 7)
    xd = on_device(x, 1)
    n = x.numel()
    buf = torch.full((n + 8,), 7.0, device="cuda")
    y = buf[1:1 + n].view(shape)
    L.cumsum_f32(xd, 1, out=y)
    L.check()
    assert buf[0].item() == 7.0 and torch.all(buf[1 + n:] == 7.0)


@pytest.mark.parametrize("op", ["sum", "mean", "max", "min", "norm"])
@pytest.mark.parametrize("shape", [(100_000, 100, 3), (4097, 5, 2), (999, 159, 3), (257, 1024, 2),
                                   (513, 33, 7), (129, 11, 256), (2000, 3, 33)])
def test_reduce(shape, op):
    L.set_option(L.OPT_COLS_VARIANT, 8)  # some of these shapes take the plane-run kernel by default
    x = inputs.make(shape, "uniform_pm1", 8)
    out = L.reduce_axis_op_f32(on_device(x), 1, op)
    L.check()
    o, n, i = shape
    if op == "sum":
        ref, scale = oracle.axis_sum(x.numpy(), o, n, i)
        assert_close(out.cpu().numpy(), ref, scale, f"planes sum {shape}")
    else:
        ref, scale = oracle.reduce_op(x.numpy(), o, n, i, op)
        assert_op_close(out, ref, scale, op, n, f"planes {op} {shape}")


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_reduce_misaligned_forced_and_exact(offset):
    shape = (6000, 100, 3)
    x = inputs.make(shape, "int:-8:8", 9)
    ref, _ = oracle.axis_sum(x.numpy(), *shape)
    got = L.reduce_axis_f32(on_device(x, offset), 1)
    assert_exact(got.cpu().numpy(), ref, f"planes sum integers at +{offset}")
    L.set_option(L.OPT_COLS_VARIANT, 8)
    shape = (100, 1500, 4)
    x = inputs.make(shape, "uniform_pm1", 10)
    ref, scale = oracle.axis_sum(x.numpy(), *shape)
    got = L.reduce_axis_f32(on_device(x, offset), 1)
    L.check()
    assert_close(got.cpu().numpy(), ref, scale, "forced planes sum")
