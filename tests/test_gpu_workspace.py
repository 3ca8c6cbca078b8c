"""The workspace variants (reduce_axis_op_ws_f32, cumsum_ws_f32): same bits as
the library-workspace calls, safe to run concurrently with separate buffers
(GPU)."""
import pytest
import torch

import oracle
from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import assert_close, bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu

REDUCE_CASES = [((1, 50_000_000), 1, "sum"), ((65536, 4096), 0, "sum"), ((65536, 4096), 0, "max"),
                ((300, 70_000), 1, "mean"), ((128, 512, 257), 1, "norm"), ((4096, 300), 1, "min"),
                ((4, 100_000, 12), 1, "sum"), ((2, 300_000, 33), 1, "mean"), ((6000, 50, 3), 1, "max")]
SCAN_CASES = [((1, 30_000_000), True, False), ((2, 5_000_000), False, True), ((512, 32768), True, False),
              ((3, 100_003), False, False)]


def garbage_ws(nbytes):
    ws = L.workspace(nbytes)
    ws.random_(0, 256)  # a reused buffer holds anything: the call must clear what matters
    return ws


@pytest.mark.parametrize("shape,dim,op", REDUCE_CASES)
def test_reduce_ws_matches_default(shape, dim, op):
    xd = on_device(inputs.make(shape, "uniform_pm1", 3))
    ref = L.reduce_axis_op_f32(xd, dim, op)
    need = L.reduce_axis_op_ws_f32(xd, dim, op)
    ws = garbage_ws(need)
    for _ in range(2):  # reuse without clearing
        got = L.reduce_axis_op_ws_f32(xd, dim, op, ws=ws)
        L.check_ws(ws)
        assert bitwise_equal(got, ref), (shape, dim, op, need)


def test_query_sizes():
    x = on_device(inputs.make((4096, 300), "uniform01", 1))
    assert L.reduce_axis_op_ws_f32(x, 1, "sum") == 256        # one warp per row: the header only
    y = on_device(inputs.make((65536, 64), "uniform01", 1))
    assert L.reduce_axis_op_ws_f32(y, 0, "sum") > 0           # split reduce axis
    nr = on_device(inputs.make((4, 100_000, 12), "uniform01", 1))
    assert L.reduce_axis_op_ws_f32(nr, 1, "sum") > 256         # narrow rows, sliced
    sp = on_device(inputs.make((6000, 50, 3), "uniform01", 1))
    assert L.reduce_axis_op_ws_f32(sp, 1, "sum") == 256        # a warp per small plane: the header only
    z = on_device(inputs.make((1, 10_000_000), "uniform01", 1))
    assert L.cumsum_ws_f32(z, 1, reverse=True) > 0            # look-back flags
    w = on_device(inputs.make((4096, 8192), "uniform01", 1))
    assert L.cumsum_ws_f32(w, 1) == 256                        # one block per row: the header only
    e = torch.empty((0, 5), device="cuda")
    assert L.cumsum_ws_f32(e, 1) == 0                          # nothing to compute


@pytest.mark.parametrize("shape,reverse,exclusive", SCAN_CASES)
def test_scan_ws_matches_default(shape, reverse, exclusive):
    xd = on_device(inputs.make(shape, "uniform01", 4))
    ref = L.cumsum_f32(xd, 1, reverse=reverse, exclusive=exclusive)
    ws = garbage_ws(L.cumsum_ws_f32(xd, 1, reverse=reverse, exclusive=exclusive))
    for _ in range(2):
        got = L.cumsum_ws_f32(xd, 1, reverse=reverse, exclusive=exclusive, ws=ws)
        L.check_ws(ws)
        assert bitwise_equal(got, ref), shape
    L.check()


def test_too_small_workspace_rejected():
    xd = on_device(inputs.make((1, 20_000_000), "uniform01", 4))
    need = L.cumsum_ws_f32(xd, 1, reverse=True)
    with pytest.raises(L.LibreduceError) as ei:
        L.cumsum_ws_f32(xd, 1, reverse=True, ws=L.workspace(need - 512))
    assert ei.value.status == L.ERR_INVALID_ARG


def test_concurrent_streams_with_separate_workspaces():
    """Four streams, each with its own workspace, run look-back scans and
    split reductions at the same time; every result matches the oracle."""
    cases = []
    for k in range(4):
        x = inputs.make((1, 4_000_000 + 4 * k), "uniform01", 10 + k)
        m = inputs.make((65536, 256), "uniform_pm1", 20 + k)
        cases.append((x, on_device(x), m, on_device(m)))
    streams = [torch.cuda.Stream() for _ in cases]
    results = []
    torch.cuda.synchronize()
    for (x, xd, m, md), st in zip(cases, streams):
        with torch.cuda.stream(st):
            ws1 = L.workspace(L.cumsum_ws_f32(xd, 1, reverse=True))
            ws2 = L.workspace(L.reduce_axis_op_ws_f32(md, 0, "sum"))
            y = L.cumsum_ws_f32(xd, 1, reverse=True, ws=ws1)
            r = L.reduce_axis_op_ws_f32(md, 0, "sum", ws=ws2)
            results.append((y, r, ws1, ws2, st))
    torch.cuda.synchronize()
    for (x, _, m, _), (y, r, ws1, ws2, st) in zip(cases, results):
        with torch.cuda.stream(st):
            L.check_ws(ws1)
            L.check_ws(ws2)
        ref, scale = oracle.reverse_cumsum(x.numpy(), 1, x.shape[1])
        assert_close(y.cpu().numpy(), ref, scale, "concurrent look-back")
        ref2, scale2 = oracle.axis_sum(m.numpy(), 1, 65536, 256)
        assert_close(r.cpu().numpy(), ref2, scale2, "concurrent split reduce")


def test_timeout_reported_through_workspace():
    xd = on_device(inputs.make((1, 8192 * 64), "uniform01", 3))
    ws = L.workspace(L.cumsum_ws_f32(xd, 1, reverse=True))
    L.set_option(L.OPT_SPIN_LIMIT, 2000)
    L.set_option(L.OPT_STALL_TILE, 5)
    L.cumsum_ws_f32(xd, 1, reverse=True, ws=ws)
    with pytest.raises(L.LibreduceError) as ei:
        L.check_ws(ws)
    assert ei.value.status == L.ERR_TIMEOUT
    L.set_option(L.OPT_STALL_TILE, -1)
    L.set_option(L.OPT_SPIN_LIMIT, 0)
    L.check_ws(ws)
    ref = L.cumsum_f32(xd, 1, reverse=True)
    assert bitwise_equal(L.cumsum_ws_f32(xd, 1, reverse=True, ws=ws), ref)


@pytest.mark.parametrize("shape,reverse,exclusive", [((2, 300_000, 4), True, False),
                                                     ((1, 5000, 4096), False, True),
                                                     ((3, 20_000, 33), True, True)])
def test_segmented_column_scan_ws_matches_default(shape, reverse, exclusive):
    """A column scan with few columns is cut into segments, whose sums and
    carries live in the caller's workspace."""
    xd = on_device(inputs.make(shape, "uniform_pm1", 5))
    ref = L.cumsum_f32(xd, 1, reverse=reverse, exclusive=exclusive)
    need = L.cumsum_ws_f32(xd, 1, reverse=reverse, exclusive=exclusive)
    assert need > 256
    ws = garbage_ws(need)
    for _ in range(2):
        got = L.cumsum_ws_f32(xd, 1, reverse=reverse, exclusive=exclusive, ws=ws)
        L.check_ws(ws)
        assert bitwise_equal(got, ref), shape
    L.check()


def test_binding_rejects_bad_out_and_workspace():
    """The workspace forms check `out` and `ws` in Python as the other
    bindings do: a wrong size, dtype, device or layout raises before any call."""
    x = on_device(inputs.make((64, 300), "uniform01", 2))
    with pytest.raises(ValueError):
        L.reduce_axis_op_ws_f32(x, 1, "sum", out=torch.empty(63, device="cuda"))
    with pytest.raises(TypeError):
        L.reduce_axis_op_ws_f32(x, 1, "sum", out=torch.empty(64, dtype=torch.float64, device="cuda"))
    with pytest.raises(ValueError):
        L.reduce_axis_op_ws_f32(x, 1, "sum", out=torch.empty(64))
    with pytest.raises(ValueError):
        L.cumsum_ws_f32(x, 1, out=torch.empty(64, 299, device="cuda"))
    with pytest.raises(ValueError):
        L.cumsum_ws_f32(x, 1, out=torch.empty(300, 64, device="cuda").t())
    with pytest.raises(ValueError):
        L.cumsum_ws_f32(x, 1, ws=torch.empty(4096, dtype=torch.uint8))
    ok = L.cumsum_ws_f32(x, 1, ws=L.workspace(L.cumsum_ws_f32(x, 1)))
    assert ok.shape == x.shape
