"""reverse_cumsum_f32 against the oracle (GPU)."""
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


def gpu_scan(x_cpu, offset=0, out_offset=0):
    xd = on_device(x_cpu, offset)
    y = on_device(torch.zeros_like(x_cpu), out_offset)
    L.reverse_cumsum_f32(xd, out=y)
    return y.cpu().numpy()


def check(rows, n, dist="uniform01", seed=3, offset=0, out_offset=0, what=""):
    x = inputs.make((rows, n), dist, seed)
    ref, scale = oracle.reverse_cumsum(x.numpy(), rows, n)
    got = gpu_scan(x, offset, out_offset)
    assert_close(got, ref, scale, what or f"[{rows},{n}] off={offset}/{out_offset}")
    assert np.array_equal(got[:, -1], x.numpy()[:, -1]) if n else True
    return got


def test_worked_examples():
    with open(os.path.join(GOLDEN, "rcumsum_worked_examples.json")) as f:
        for c in json.load(f)["cases"]:
            x = torch.tensor([c["x"]], dtype=torch.float32)
            assert gpu_scan(x).reshape(-1).tolist() == [float(v) for v in c["y"]]


N_LIST = [1, 2, 3, 4, 31, 32, 33, 1023, 1024, 1025, 4095, 4096, 4097, 8191, 8192, 8193, 32768, 100003]


@pytest.mark.parametrize("n", N_LIST)
@pytest.mark.parametrize("rows", [1, 2, 3, 37])
def test_shapes(rows, n):
    check(rows, n, dist="uniform_pm1")


@pytest.mark.parametrize("offset,out_offset", [(1, 0), (0, 3), (2, 2), (3, 1)])
def test_misaligned(offset, out_offset):
    check(5, 8192, offset=offset, out_offset=out_offset)
    check(3, 1001, offset=offset, out_offset=out_offset)


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("shape", [(7, 4096), (3, 12288), (2, 32768), (9, 100), (4, 50000)])
def test_variants(variant, shape):
    L.set_option(L.OPT_SCAN_STRATEGY, 1)  # one block per row, whatever the row count
    L.set_option(L.OPT_RSCAN_VARIANT, variant)
    check(*shape, what=f"variant {variant} {shape}")


@pytest.mark.parametrize("shape", [(64, 32768), (3, 100001), (1000, 37)])
def test_integer_inputs_exact(shape):
    x = inputs.make(shape, "int:0:3", 3)
    ref, _ = oracle.reverse_cumsum(x.numpy(), *shape)
    assert_exact(gpu_scan(x), ref, f"int {shape}")


def test_long_row_accuracy():
    # Many tiles per row: the carry chain is blocked, the tolerance still holds.
    check(2, 3_000_001, dist="uniform01", seed=8)


def test_deterministic_bitwise():
    xd = on_device(inputs.make((256, 32768), "uniform01", 3))
    outs = [L.reverse_cumsum_f32(xd).clone() for _ in range(3)]
    for o in outs[1:]:
        assert bitwise_equal(outs[0], o)


def test_nan_inf():
    x = inputs.make((3, 5000), "uniform01", 1)
    x[1, 2500] = float("nan")
    x[2, 100] = float("inf")
    got = gpu_scan(x)
    assert np.isnan(got[1, :2501]).all() and np.isfinite(got[1, 2501:]).all()
    assert (got[2, :101] == np.inf).all() and np.isfinite(got[2, 101:]).all()
    assert np.isfinite(got[0]).all()
