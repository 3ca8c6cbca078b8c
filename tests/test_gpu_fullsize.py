"""The five workloads at full size, in the launch configuration bench.py times
(default options), against the oracle on EVERY output (GPU).

For each workload:
  * the seeded float input is compared with the oracle within the tolerance
    |gpu - ref| <= 1e-5 * sum|x| + 1e-6 per output;
  * the integer-valued variant ({-1, 0, 1} for the 1D sums, [-8, 8] for the
    axis sums, {0..3} for the scan) must equal the oracle exactly;
  * three runs give bit-identical outputs.

The oracle is single-threaded C; to keep the checks to seconds the test runs it
on independent pieces of the output (ranges of output positions, blocks of
rows) from a thread pool.  ctypes releases the GIL during the call, so the
pieces run in parallel on the host cores.  Each piece is the oracle's own
definition on its own outputs; nothing is reordered inside an output.
"""
import concurrent.futures
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_common import libreduce_defaults  # noqa: F401
from parity import assert_close, assert_exact, bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda", 0)
WORKERS = max(1, min(32, len(os.sched_getaffinity(0))))


def workload(name, dist=None):
    w = dict(inputs.WORKLOADS[name])
    if dist:
        w["dist"] = dist
    return w, inputs.make(w["shape"], w["dist"], w["seed"], device=DEV)


def pmap(fn, items):
    with concurrent.futures.ThreadPoolExecutor(WORKERS) as ex:
        return list(ex.map(fn, items))


def three_runs(call):
    """Run `call` three times; assert the outputs are bit-identical; return one."""
    outs = [call().clone() for _ in range(3)]
    L.check()
    assert bitwise_equal(outs[0], outs[1]) and bitwise_equal(outs[0], outs[2]), "reruns differ"
    return outs[0]


def axis_all_outputs(xh, outer, reduce, inner):
    """The oracle's axis sum at every output, positions split over threads."""
    n_out = outer * inner
    bounds = np.linspace(0, n_out, 4 * WORKERS + 1).astype(np.int64)

    def piece(k):
        pos = np.arange(bounds[k], bounds[k + 1], dtype=np.int64)
        return oracle.axis_sum_at(xh, outer, reduce, inner, pos)

    parts = pmap(piece, range(len(bounds) - 1))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def check(got, ref, scale, integer, what):
    if integer:
        assert_exact(got, ref, what)
    else:
        assert_close(got, ref, scale, what)


# ---- configs 1 and 2: the 1D sum --------------------------------------------------------

@pytest.mark.parametrize("name", ["sum_1e6_harmonic", "sum_1e6_pm1"])
def test_sum_1e6(name):
    w, x = workload(name)
    s = three_runs(lambda: L.reduce_sum_f32(x))
    ref, scale = oracle.sum1d(x.cpu().numpy())
    assert_close(s.item(), ref, scale, name)


def test_sum_1e6_integers():
    x = inputs.make((1_000_000,), "int:-1:1", 42, device=DEV)
    s = three_runs(lambda: L.reduce_sum_f32(x))
    ref, _ = oracle.sum1d(x.cpu().numpy())
    assert_exact(s.item(), ref, "sum 1e6 {-1,0,1}")


@pytest.mark.parametrize("n", inputs.SUM_SWEEP)
@pytest.mark.parametrize("dist", ["uniform01", "int:-1:1"])
def test_sum_sweep(n, dist):
    """Every size of the sweep, seeded uniform[0,1) and {-1, 0, 1}.  For the
    integer input every partial sum is an integer; it stays below 2^24 for any
    n < 2^24, and at 5e8 and 1e9 the partials are sums of independent
    {-1, 0, 1} terms, whose spread (about sqrt(2n/3) < 26,000) is far below
    2^24, so the sum is exact except with negligible probability."""
    x = inputs.make((n,), dist, 42, device=DEV)
    s = three_runs(lambda: L.reduce_sum_f32(x))
    ref, scale = oracle.sum1d(x.cpu().numpy())
    check(s.item(), ref, scale, dist.startswith("int"), f"sum {n} {dist}")


# ---- config 3: [128, 4096, 4095] over dim 1 ------------------------------------------

@pytest.mark.parametrize("dist", [None, "int:-8:8"])
def test_axis_128x4096x4095(dist):
    w, x = workload("axis_128x4096x4095_d1", dist)
    out = three_runs(lambda: L.reduce_axis_f32(x, 1)).cpu().numpy().reshape(-1)
    xh = x.cpu().numpy()
    del x
    ref, scale = axis_all_outputs(xh, 128, 4096, 4095)
    check(out, ref, scale, dist is not None, "axis cfg3")


# ---- config 4: [4096, 65536] over dim 1 and [65536, 4096] over dim 0 ---------------

@pytest.mark.parametrize("dist", [None, "int:-8:8"])
def test_axis_4096x65536_d1(dist):
    w, x = workload("axis_4096x65536_d1", dist)
    out = three_runs(lambda: L.reduce_axis_f32(x, 1)).cpu().numpy()
    ref, scale = axis_all_outputs(x.cpu().numpy(), 4096, 65536, 1)
    check(out, ref, scale, dist is not None, "axis 4a")


@pytest.mark.parametrize("dist", [None, "int:-8:8"])
def test_axis_65536x4096_d0(dist):
    w, x = workload("axis_65536x4096_d0", dist)
    out = three_runs(lambda: L.reduce_axis_f32(x, 0)).cpu().numpy()
    ref, scale = axis_all_outputs(x.cpu().numpy(), 1, 65536, 4096)
    check(out, ref, scale, dist is not None, "axis 4b")


# ---- config 5: reverse cumsum of [32768, 32768] -----------------------------------

def rows_all_outputs(xh, yh, rows, n, integer, what, block=256):
    """Reverse scan of every row by the oracle, blocks of rows over threads,
    each block compared with the GPU output as it is produced."""
    def piece(r0):
        r1 = min(rows, r0 + block)
        ref, scale = oracle.reverse_cumsum(xh[r0:r1], r1 - r0, n)
        check(yh[r0:r1], ref, scale, integer, f"{what} rows {r0}..{r1 - 1}")

    pmap(piece, range(0, rows, block))


@pytest.mark.parametrize("dist", [None, "int:0:3"])
def test_rcumsum_32768x32768(dist):
    w, x = workload("rcumsum_32768x32768", dist)
    y = three_runs(lambda: L.reverse_cumsum_f32(x))
    assert torch.equal(y[:, -1], x[:, -1])  # the last column is x itself, no additions
    rows_all_outputs(x.cpu().numpy(), y.cpu().numpy(), 32768, 32768, dist is not None, "rcumsum cfg5")


# ---- one row of 1e9: the decoupled look-back --------------------------------------

@pytest.mark.parametrize("dist", [None, "int:0:3"])
def test_rcumsum_1x1e9_lookback(dist):
    """The bench's [1, 1e9] reverse scan (float4 look-back, aligned, 122,071
    tiles: four levels of the 32-ary tree) against the oracle on every
    output.  For the {0..3} input the long suffixes (up to about 1.5e9)
    exceed 2^24, where fp32 no longer holds every integer, so that run is
    compared within the tolerance everywhere, and exactly on the last
    4,194,304 outputs: each of their suffixes, and every partial sum that
    forms one, is an integer of at most 3 * 2^22 < 2^24."""
    w, x = workload("rcumsum_1x1e9", dist)
    n = w["shape"][1]
    y = three_runs(lambda: L.reverse_cumsum_f32(x))
    xh = x.cpu().numpy().reshape(-1)
    yh = y.cpu().numpy().reshape(-1)
    del x, y
    ref, scale = oracle.reverse_cumsum(xh, 1, n)
    ref, scale = ref.reshape(-1), scale.reshape(-1)
    step = 10_000_000

    def piece(j0):
        j1 = min(n, j0 + step)
        assert_close(yh[j0:j1], ref[j0:j1], scale[j0:j1], f"1e9 row [{j0}, {j1})")

    pmap(piece, range(0, n, step))
    assert yh[-1] == xh[-1]
    if dist is not None:
        tail = 4_194_304  # every suffix here is an integer <= 3 * 2^22 < 2^24
        assert_exact(yh[-tail:], ref[-tail:], "1e9 row, integer tail")
