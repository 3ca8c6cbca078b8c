"""The single-pass look-back reverse scan (few long rows) against the oracle,
its bit-identity across runs, and its bounded waits (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import assert_close, assert_exact, bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu
LOOKBACK = 2


def run(x_cpu, offset=0, out_offset=0):
    xd = on_device(x_cpu, offset)
    y = on_device(torch.zeros_like(x_cpu), out_offset)
    L.reverse_cumsum_f32(xd, out=y)
    L.check()
    return y.cpu().numpy()


def check(rows, n, dist="uniform01", seed=3, offset=0, out_offset=0, force=True):
    if force:
        L.set_option(L.OPT_SCAN_STRATEGY, LOOKBACK)
    x = inputs.make((rows, n), dist, seed)
    ref, scale = oracle.reverse_cumsum(x.numpy(), rows, n)
    got = run(x, offset, out_offset)
    assert_close(got, ref, scale, f"look-back [{rows},{n}] off={offset}/{out_offset}")
    assert np.array_equal(got[:, -1], x.numpy()[:, -1])


@pytest.mark.parametrize("n", [1, 100, 8191, 8192, 8193, 3 * 65536 + 5, 1_000_003, 2 ** 24])
def test_one_row(n):
    check(1, n, dist="uniform_pm1")


@pytest.mark.parametrize("rows,n", [(2, 32768), (3, 100003), (7, 65536), (31, 8192 * 9 + 4)])
def test_few_rows(rows, n):
    check(rows, n)


@pytest.mark.parametrize("offset,out_offset", [(1, 0), (0, 2), (3, 3)])
def test_misaligned_scalar_path(offset, out_offset):
    check(2, 300_001, offset=offset, out_offset=out_offset)
    check(1, 77_777, offset=offset, out_offset=out_offset)


def test_auto_dispatch_few_rows():
    # One long row is sent to the look-back scan without any option.
    check(1, 5_000_000, force=False)
    check(3, 2_000_000, force=False)


def test_integer_inputs_exact():
    L.set_option(L.OPT_SCAN_STRATEGY, LOOKBACK)
    x = inputs.make((1, 1 << 22), "int:0:3", 3)
    ref, _ = oracle.reverse_cumsum(x.numpy(), 1, 1 << 22)
    assert_exact(run(x), ref, "look-back int")


def test_deterministic_bitwise():
    L.set_option(L.OPT_SCAN_STRATEGY, LOOKBACK)
    xd = on_device(inputs.make((1, 1 << 25), "uniform01", 3))
    outs = [L.reverse_cumsum_f32(xd).clone() for _ in range(3)]
    L.check()
    for o in outs[1:]:
        assert bitwise_equal(outs[0], o)


def test_matches_block_per_row_path():
    # Same data through every strategy: all within tolerance of the oracle.
    x = inputs.make((4, 123_456), "uniform01", 9)
    ref, scale = oracle.reverse_cumsum(x.numpy(), 4, 123_456)
    for strategy in (1, 2, 3, 4):
        L.set_option(L.OPT_SCAN_STRATEGY, strategy)
        assert_close(run(x), ref, scale, f"strategy {strategy}")


@pytest.mark.parametrize("lag", [1, 7, 64, 768, 5000])
def test_lag_values(lag):
    # Any lag gives a correct result (a small one only waits more, a large one
    # rereads from HBM instead of L2).
    L.set_option(L.OPT_LOOKBACK_LAG, lag)
    check(2, 8192 * 300 + 4)


@pytest.mark.parametrize("strategy", [2, 3, 4])
@pytest.mark.parametrize("n", [8192 * 6 * 152 + 8, 8192 * 40000])
def test_long_rows_both_forms(n, strategy):
    L.set_option(L.OPT_SCAN_STRATEGY, strategy)
    check(1, n, force=False)


def test_bounded_wait_reports_timeout():
    """A tile that never publishes (a fault chosen on the host) makes the waits
    behind it run out; the kernel returns, the host reads TIMEOUT, and the
    library keeps working afterwards."""
    x = on_device(inputs.make((1, 8192 * 64), "uniform01", 3))
    L.set_option(L.OPT_SCAN_STRATEGY, LOOKBACK)
    L.set_option(L.OPT_SPIN_LIMIT, 2000)
    L.set_option(L.OPT_STALL_TILE, 5)
    for strategy in (2, 3):  # L2-lag form and one tile per block
        L.set_option(L.OPT_SCAN_STRATEGY, strategy)
        L.reverse_cumsum_f32(x)
        with pytest.raises(L.LibreduceError) as ei:
            L.check()
        assert ei.value.status == L.ERR_TIMEOUT
    L.set_option(L.OPT_STALL_TILE, -1)
    L.set_option(L.OPT_SPIN_LIMIT, 0)
    L.check()  # the error word was cleared
    xc = x.cpu()
    ref, scale = oracle.reverse_cumsum(xc.numpy(), 1, xc.shape[1])
    assert_close(L.reverse_cumsum_f32(x).cpu().numpy(), ref, scale, "after timeout")


@pytest.mark.parametrize("rows,n", [(1, 1), (1, 8191), (2, 8193), (3, 100_003), (1, 2_000_001)])
def test_reduce_then_scan_shapes(rows, n):
    L.set_option(L.OPT_SCAN_STRATEGY, 4)
    check(rows, n, force=False)


def test_reduce_then_scan_deterministic():
    L.set_option(L.OPT_SCAN_STRATEGY, 4)
    xd = on_device(inputs.make((2, 5_000_000), "uniform01", 7))
    a = L.reverse_cumsum_f32(xd).clone()
    b = L.reverse_cumsum_f32(xd).clone()
    assert bitwise_equal(a, b)
