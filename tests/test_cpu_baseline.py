"""The all-core CPU baseline that bench.py reports beside the oracle: fp64
sums over independent outputs or segments, fp32 results.  Checked against
numpy's fp64 sums; each output may differ only by its final fp32 rounding
(plus a few fp64 ulps from the order of the segment sums)."""
import numpy as np
import pytest

import cpu_baseline as cb


def close32(got, ref):
    ref = np.asarray(ref, np.float64)
    tol = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) + 1e-9 * np.abs(ref)
    assert np.all(np.abs(np.asarray(got, np.float64) - ref) <= tol)


@pytest.mark.parametrize("threads", [1, 3, 8])
def test_sum(threads):
    x = np.random.default_rng(0).standard_normal(1_000_003).astype(np.float32)
    close32(cb.sum1d(x, threads), np.sum(x, dtype=np.float64))
    assert cb.sum1d(np.zeros(0, np.float32), threads) == 0.0


@pytest.mark.parametrize("shape", [(5, 777, 1), (3, 129, 300), (1, 1000, 513), (2, 0, 7)])
def test_axis_sum(shape):
    x = np.random.default_rng(1).random(shape, dtype=np.float32)
    close32(cb.axis_sum(x, *shape, threads=4), x.astype(np.float64).sum(axis=1))


@pytest.mark.parametrize("rows,n,threads", [(9, 1001, 4), (1, 100_003, 6), (2, 50_001, 5), (1, 7, 16)])
def test_reverse_cumsum(rows, n, threads):
    x = np.random.default_rng(2).random((rows, n), dtype=np.float32)
    ref = np.flip(np.cumsum(np.flip(x.astype(np.float64), 1), 1), 1)
    close32(cb.reverse_cumsum(x, rows, n, threads), ref)


def test_reports_cores_and_model():
    assert cb.cores() >= 1
    assert isinstance(cb.cpu_model(), str) and cb.cpu_model()
