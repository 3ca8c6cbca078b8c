"""The follow-on workloads (other scan forms, other reductions, caller
scratch) at the full sizes bench.py times, with default options, against the
oracle: sampled outputs, always with the edges, where the oracle cannot take
the whole output in seconds (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import libreduce_defaults  # noqa: F401
from parity import assert_close, assert_op_close, bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda", 0)


def workload(name):
    w = dict(inputs.WORKLOADS[name])
    return w, inputs.make(w["shape"], w["dist"], w["seed"], device=DEV)


def pick(n, k, seed, edges=(0, 1, 31, 32, 1023, 1024)):
    rng = np.random.default_rng(seed)
    base = [e for e in edges if e < n] + [n // 2, n - 2, n - 1]
    return np.unique(np.clip(np.concatenate([base, rng.integers(0, n, k)]), 0, n - 1))


def column_scan_check(name, ocount=6, icount=24):
    """Scan along dim 1 of [outer, N, inner]: whole columns at sampled (o, i),
    gathered into [len(o), N, len(i)] and scanned by the oracle."""
    w, x = workload(name)
    outer, n, inner = w["shape"]
    y = L.cumsum_f32(x, 1, reverse=w["reverse"], exclusive=w["exclusive"])
    L.check()
    os_ = torch.as_tensor(pick(outer, ocount, 1, edges=(0, 1)), device=DEV)
    is_ = torch.as_tensor(pick(inner, icount, 2, edges=(0, 1, 63, 64, 255, 256)), device=DEV)
    xs = x.index_select(0, os_).index_select(2, is_).contiguous().cpu().numpy()
    ys = y.index_select(0, os_).index_select(2, is_).cpu().numpy()
    ref, scale = oracle.cumsum(xs, len(os_), n, len(is_), w["reverse"], w["exclusive"])
    assert_close(ys, ref, scale, name)


def test_cumsum_fwd_32768x32768():
    w, x = workload("cumsum_fwd_32768x32768")
    y = L.cumsum_f32(x, 1)
    assert torch.equal(y[:, 0], x[:, 0])  # the first output of a forward inclusive scan is x
    rows = torch.as_tensor(pick(32768, 40, 3, edges=(0, 1)), device=DEV)
    xs = x.index_select(0, rows).cpu().numpy()
    ref, scale = oracle.cumsum(xs, len(rows), 32768, 1, False, False)
    assert_close(y.index_select(0, rows).cpu().numpy(), ref, scale, "forward rows")


def test_cumsum_fwd_excl_1e9():
    """One row of 1e9, forward exclusive (look-back): y[j] = sum of x[:j], the
    oracle's sum of each sampled prefix."""
    w, x = workload("cumsum_fwd_excl_1x1e9")
    n = w["shape"][1]
    y = L.cumsum_f32(x, 1, exclusive=True)
    L.check()
    assert y[0, 0].item() == 0.0
    xh = x.cpu().numpy().reshape(-1)
    js = np.concatenate([[1, 2, 4096, 4097], pick(n, 4, 4)[1:]])
    got = y[0, torch.as_tensor(js, device=DEV)].cpu().numpy()
    for j, g in zip(js, got):
        ref, scale = oracle.sum1d(xh[:j])
        assert_close(g, ref, scale, f"prefix {j}")


def test_rcumsum_1e9_reduce_then_scan():
    """The same long row as three passes (tile sums, their scan, the carried
    rescan): sampled suffix sums from the oracle, and the last output is x."""
    w, x = workload("rcumsum_1x1e9_rts")
    n = w["shape"][1]
    L.set_option(L.OPT_SCAN_STRATEGY, w["strategy"])
    y = L.reverse_cumsum_f32(x)
    L.check()
    assert y[0, -1].item() == x[0, -1].item()
    xh = x.cpu().numpy().reshape(-1)
    js = np.concatenate([[0, n - 4097, n - 2], pick(n, 3, 5)[1:-1]])
    got = y[0, torch.as_tensor(js, device=DEV)].cpu().numpy()
    for j, g in zip(js, got):
        ref, scale = oracle.sum1d(xh[j:])
        assert_close(g, ref, scale, f"suffix {j}")


@pytest.mark.parametrize("name", ["cumsum_128x4096x4095_d1", "cumsum_64x16384x1024_d1",
                                  "cumsum_2x8192x4096_d1", "cumsum_1024x8192x64_d1"])
def test_column_scans(name):
    column_scan_check(name)


def test_max_1e9():
    w, x = workload("max_1e9")
    got = L.reduce_f32(x, "max").item()
    ref, scale = oracle.reduce_op(x.cpu().numpy(), 1, w["shape"][0], 1, "max")
    assert_op_close(np.array([got]), ref, scale, "max", w["shape"][0], "max 1e9")


@pytest.mark.parametrize("name", ["norm_128x4096x4095_d1", "mean_4096x65536_d1", "min_65536x4096_d0",
                                  "sum_16x1000000x12_d1"])
def test_axis_ops(name):
    w, x = workload(name)
    outer, r, inner = L.canonical_axis(w["shape"], w["dim"])
    out = L.reduce_axis_op_f32(x, w["dim"], w["rop"]).reshape(outer, inner)
    if w["rop"] == "sum":  # the sum's oracle and tolerance
        ref, scale = oracle.axis_sum(x.cpu().numpy(), outer, r, inner)
        assert_close(out.cpu().numpy(), ref, scale, name)
        return
    if outer * r * inner <= 300_000_000:
        ref, scale = oracle.reduce_op(x.cpu().numpy(), outer, r, inner, w["rop"])
        assert_op_close(out, ref, scale, w["rop"], r, name)
        return
    # [128, 4096, 4095]: whole columns at sampled (o, i).
    x3 = x.view(outer, r, inner)
    os_ = torch.as_tensor(pick(outer, 6, 6, edges=(0, 1)), device=DEV)
    is_ = torch.as_tensor(pick(inner, 40, 7), device=DEV)
    xs = x3.index_select(0, os_).index_select(2, is_).contiguous().cpu().numpy()
    ref, scale = oracle.reduce_op(xs, len(os_), r, len(is_), w["rop"])
    got = out.index_select(0, os_).index_select(1, is_)
    assert_op_close(got, ref, scale, w["rop"], r, name)


def test_workspace_calls_match_default():
    """The caller-scratch forms give the same bits as the library-scratch
    calls at full size."""
    w, x = workload("rcumsum_1x1e9_ws")
    ref = L.cumsum_f32(x, 1, reverse=True)
    ws = L.workspace(L.cumsum_ws_f32(x, 1, reverse=True))
    got = L.cumsum_ws_f32(x, 1, reverse=True, ws=ws)
    L.check_ws(ws)
    assert bitwise_equal(got, ref)
    del x, ref, got, ws
    w, x = workload("axis_65536x4096_d0_ws")
    ref = L.reduce_axis_op_f32(x, 0, "sum")
    ws = L.workspace(L.reduce_axis_op_ws_f32(x, 0, "sum"))
    got = L.reduce_axis_op_ws_f32(x, 0, "sum", ws=ws)
    L.check_ws(ws)
    assert bitwise_equal(got, ref)


def offset_pair(shape, offset, dist, seed):
    """x and y of `shape` at the same 4-byte offset from 16-byte aligned
    allocations, x filled from the seeded generator."""
    n = int(np.prod(shape))
    xb = torch.empty(n + 4, dtype=torch.float32, device=DEV)
    yb = torch.empty(n + 4, dtype=torch.float32, device=DEV)
    x = xb[offset:offset + n].view(shape)
    x.copy_(inputs.make(shape, dist, seed, device=DEV))
    return x, yb[offset:offset + n].view(shape)


@pytest.mark.parametrize("offset", [0, 1])
def test_odd_long_row_both_directions(offset):
    """One row of 999,999,999 (not a whole number of float4s), at a 4-byte
    offset or not: the float4 look-back with masked row edges, reverse and
    forward exclusive, against the oracle's sums of sampled suffixes and
    prefixes; the end outputs are exact."""
    n = 999_999_999
    x, y = offset_pair((1, n), offset, "uniform01", 23)
    xh = x.cpu().numpy().reshape(-1)
    js = pick(n, 3, 6, edges=(0, 1, 2, 3, 4, 4095, 4096, 8191, 8192))
    L.reverse_cumsum_f32(x, out=y)
    L.check()
    assert y[0, -1].item() == x[0, -1].item()
    got = y[0, torch.as_tensor(js, device=DEV)].cpu().numpy()
    for j, g in zip(js, got):
        ref, scale = oracle.sum1d(xh[j:])
        assert_close(g, ref, scale, f"suffix {j} (offset {offset})")
    L.cumsum_f32(x, 1, exclusive=True, out=y)
    L.check()
    assert y[0, 0].item() == 0.0
    got = y[0, torch.as_tensor(js, device=DEV)].cpu().numpy()
    for j, g in zip(js, got):
        ref, scale = oracle.sum1d(xh[:j])
        assert_close(g, ref, scale, f"prefix {j} (offset {offset})")


@pytest.mark.parametrize("reverse", [True, False])
def test_odd_rows_at_offset(reverse):
    """[32768, 32767] at a 4-byte offset: one block per row with masked row
    edges.  Sampled rows against the oracle, the end column exactly x."""
    x, y = offset_pair((32768, 32767), 3, "uniform01", 29)
    L.cumsum_f32(x, 1, reverse=reverse, out=y)
    L.check()
    end = -1 if reverse else 0
    assert torch.equal(y[:, end], x[:, end])
    rows = torch.as_tensor(pick(32768, 40, 7, edges=(0, 1, 2, 3)), device=DEV)
    xs = x.index_select(0, rows).cpu().numpy()
    ref, scale = oracle.cumsum(xs, len(rows), 32767, 1, reverse, False)
    assert_close(y.index_select(0, rows).cpu().numpy(), ref, scale, f"odd rows reverse={reverse}")


def test_short_rows_full_size():
    """The two short-row workloads of the bench, in its launch configuration:
    sampled rows of the reverse scan of [2e6, 100] and of the row sums of
    [4e6, 32] against the oracle; the scan's last column is exactly x."""
    w, x = workload("rcumsum_2000000x100")
    rows, n = w["shape"]
    y = L.cumsum_f32(x, 1, reverse=True)
    L.check()
    assert torch.equal(y[:, -1], x[:, -1])
    pick_rows = torch.as_tensor(pick(rows, 60, 8, edges=(0, 1, 2, 63, 64)), device=DEV)
    ref, scale = oracle.cumsum(x.index_select(0, pick_rows).cpu().numpy(), len(pick_rows), n, 1, True, False)
    assert_close(y.index_select(0, pick_rows).cpu().numpy(), ref, scale, "short rows scan")
    w, x = workload("sum_4000000x32_d1")
    rows, n = w["shape"]
    s = L.reduce_axis_f32(x, 1)
    L.check()
    ref, scale = oracle.axis_sum(x.cpu().numpy(), rows, n, 1)
    assert_close(s.cpu().numpy(), ref[:, 0], scale[:, 0], "short rows sum")


@pytest.mark.parametrize("name", ["cumsum_100000x100x3_d1", "cumsum_4096x4096x2_d1", "cumsum_1x40000000x4_d1",
                                  "cumsum_100000x100x16_d1"])
def test_narrow_plane_scans_every_output(name):
    """The bench's narrow-plane scans at full size, every output against the
    oracle, and a rerun bit for bit."""
    w, x = workload(name)
    outer, n, inner = w["shape"]
    y = L.cumsum_f32(x, 1, reverse=w["reverse"], exclusive=w["exclusive"]).clone()
    again = L.cumsum_f32(x, 1, reverse=w["reverse"], exclusive=w["exclusive"])
    L.check()
    assert bitwise_equal(y, again)
    ref, scale = oracle.cumsum(x.cpu().numpy(), outer, n, inner, w["reverse"], w["exclusive"])
    assert_close(y.cpu().numpy(), ref, scale, name)


def test_narrow_plane_sum_every_output():
    w, x = workload("sum_100000x100x3_d1")
    outer, n, inner = w["shape"]
    out = L.reduce_axis_op_f32(x, 1, "sum")
    L.check()
    ref, scale = oracle.axis_sum(x.cpu().numpy(), outer, n, inner)
    assert_close(out.cpu().numpy(), ref, scale, "sum [100000, 100, 3]")
