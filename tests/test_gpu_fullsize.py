"""The five workloads at full size, in the launch configuration bench.py times
(default options), against the oracle: every output where the oracle is
cheap, sampled outputs (with all edges) where it is not (GPU)."""
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


def workload(name, dist=None):
    w = dict(inputs.WORKLOADS[name])
    if dist:
        w["dist"] = dist
    return w, inputs.make(w["shape"], w["dist"], w["seed"], device=DEV)


def sample_positions(outer, inner, m, seed):
    rng = np.random.default_rng(seed)
    edge_i = np.unique(np.clip([0, 1, 31, 32, 63, 64, 127, 128, 255, 256, 1023, 1024, inner - 2, inner - 1],
                               0, inner - 1))
    edge_o = np.unique(np.clip([0, 1, outer // 2, outer - 1], 0, outer - 1))
    pos = [o * inner + i for o in edge_o for i in edge_i]
    pos += list(rng.integers(0, outer * inner, m))
    return np.unique(np.asarray(pos, dtype=np.int64))


def test_sum_1e9():
    w, x = workload("sum_1e9")
    s = L.reduce_sum_f32(x).item()
    ref, scale = oracle.sum1d(x.cpu().numpy())
    assert_close(s, ref, scale, "sum 1e9")
    again = [L.reduce_sum_f32(x).clone() for _ in range(2)]
    assert bitwise_equal(again[0], again[1])


@pytest.mark.parametrize("n", [500_000_000])
def test_sum_5e8(n):
    x = inputs.make((n,), "uniform01", 42, device=DEV)
    ref, scale = oracle.sum1d(x.cpu().numpy())
    assert_close(L.reduce_sum_f32(x).item(), ref, scale, "sum 5e8")


@pytest.mark.parametrize("dist", [None, "int:-8:8"])
def test_axis_128x4096x4095(dist):
    w, x = workload("axis_128x4096x4095_d1", dist)
    out = L.reduce_axis_f32(x, 1).cpu().numpy().reshape(-1)
    xh = x.cpu().numpy()
    del x
    pos = sample_positions(128, 4095, 1500, 7)
    ref, scale = oracle.axis_sum_at(xh, 128, 4096, 4095, pos)
    if dist:
        assert_exact(out[pos], ref, "axis cfg3 int")
    else:
        assert_close(out[pos], ref, scale, "axis cfg3")


def test_axis_4096x65536_d1():
    w, x = workload("axis_4096x65536_d1")
    out = L.reduce_axis_f32(x, 1).cpu().numpy()
    ref, scale = oracle.axis_sum(x.cpu().numpy(), 4096, 65536, 1)
    assert_close(out, ref[:, 0], scale[:, 0], "axis 4a")


def test_axis_65536x4096_d0():
    w, x = workload("axis_65536x4096_d0")
    out = L.reduce_axis_f32(x, 0).cpu().numpy()
    pos = sample_positions(1, 4096, 600, 11)
    ref, scale = oracle.axis_sum_at(x.cpu().numpy(), 1, 65536, 4096, pos)
    assert_close(out[pos], ref, scale, "axis 4b")


@pytest.mark.parametrize("dist", [None, "int:0:3"])
def test_rcumsum_32768x32768(dist):
    w, x = workload("rcumsum_32768x32768", dist)
    y = L.reverse_cumsum_f32(x)
    # Every row: the last column is x itself, the first is the row sum.
    assert torch.equal(y[:, -1], x[:, -1])
    first = y[:, 0].cpu().numpy()
    xh = x.cpu().numpy()
    rows_ref, rows_scale = oracle.axis_sum(xh, 32768, 32768, 1)
    assert_close(first, rows_ref[:, 0], rows_scale[:, 0], "rcumsum first column")
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 1, 16383, 32766, 32767], rng.integers(0, 32768, 40)]))
    yh = y[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    sub = np.ascontiguousarray(xh[rows])
    ref, scale = oracle.reverse_cumsum(sub, len(rows), 32768)
    if dist:
        assert_exact(yh, ref, "rcumsum int rows")
    else:
        assert_close(yh, ref, scale, "rcumsum rows")


def test_rcumsum_one_long_row():
    """Few long rows take the look-back scan by default."""
    n = 200_000_000
    x = inputs.make((1, n), "uniform01", 5, device=DEV)
    y = L.reverse_cumsum_f32(x)
    L.check()
    ref, scale = oracle.reverse_cumsum(x.cpu().numpy(), 1, n)
    assert_close(y.cpu().numpy(), ref, scale, "one row of 2e8")
