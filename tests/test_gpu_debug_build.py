"""One parity run of the debug build on the GPU: a call of each kernel family
through libreduce_debug.so, whose device-side checks skip and report any
access outside the call's buffers.  Every output matches the oracle and the
checks find nothing (libreduce_check returns OK).  The debug build never
takes the single-pass column look-back (its checked form faulted, cause
unknown); the [2, 8192, 4096] case runs the three-pass column scan there."""
import ctypes

import pytest
import torch

import oracle
from gpu_common import on_device
from parity import assert_close
from reduction_scan_primitives_gb300 import build as lib_build
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    return L.load(lib_build.build(debug=True))


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def check(dbg):
    st = dbg.libreduce_check(stream())
    assert st == L.OK, (st, hex(dbg.libreduce_debug_bad_address()))


@pytest.mark.parametrize("n", [1, 10_003, 100_001, 3_000_001])
def test_sum(dbg, n):
    x = on_device(inputs.make((n,), "uniform_pm1", 31), offset=n % 4)
    out = torch.empty((), device="cuda")
    assert dbg.reduce_sum_f32(ptr(x), n, ptr(out), stream()) == L.OK
    check(dbg)
    ref, scale = oracle.sum1d(x.cpu().numpy())
    assert_close(out.item(), ref, scale, f"debug sum {n}")
    assert dbg.reduce_sum_f32_noalloc(ptr(x), n, ptr(out), stream()) == L.OK
    check(dbg)
    assert_close(out.item(), ref, scale, f"debug noalloc sum {n}")


@pytest.mark.parametrize("shape", [(37, 513, 67), (64, 40_000, 1), (3000, 100, 1), (5, 1000, 12),
                                   (20_000, 100, 3), (2, 300_000, 64), (30_000, 101, 5),
                                   (3000, 99, 11), (4000, 35, 17), (1000, 300, 40), (60_000, 40, 20)])
def test_axis_sum(dbg, shape):
    x = on_device(inputs.make(shape, "uniform_pm1", 32))
    o, r, i = shape
    out = torch.empty(o * i, device="cuda")
    assert dbg.reduce_axis_f32(ptr(x), o, r, i, ptr(out), stream()) == L.OK
    check(dbg)
    ref, scale = oracle.axis_sum(x.cpu().numpy(), o, r, i)
    assert_close(out.cpu().numpy(), ref, scale, f"debug axis {shape}")


@pytest.mark.parametrize("shape,flags", [((33, 10_000, 1), 1), ((2, 600_001, 1), 1), ((5001, 100, 1), 0),
                                         ((1, 3_000_000, 1), 3), ((8, 1000, 12), 2), ((2, 8192, 4096), 2),
                                         ((20_000, 100, 3), 1), ((64, 4096, 2), 0), ((1, 400_000, 2), 1),
                                         ((3, 7000, 4095), 0), ((100_000, 7, 3), 2), ((30_000, 101, 5), 0),
                                         ((2, 300_000, 3), 0), ((2, 300_000, 3), 3),
                                         ((3000, 101, 13), 1), ((700, 1001, 15), 2), ((2000, 50, 34), 0),
                                         ((100, 2000, 100), 3), ((20_000, 100, 16), 0), ((60_000, 40, 20), 1)])
def test_cumsum(dbg, shape, flags):
    x = on_device(inputs.make(shape, "uniform01", 33))
    y = torch.empty_like(x)
    o, n, i = shape
    assert dbg.cumsum_f32(ptr(x), o, n, i, ptr(y), flags, stream()) == L.OK
    check(dbg)
    ref, scale = oracle.cumsum(x.cpu().numpy(), o, n, i, bool(flags & 1), bool(flags & 2))
    assert_close(y.cpu().numpy(), ref, scale, f"debug cumsum {shape} flags {flags}")
