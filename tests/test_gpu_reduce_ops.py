"""reduce_f32 / reduce_axis_op_f32 (mean, max, min, norm) against the oracle
(GPU).  Sum is covered by test_gpu_sum / test_gpu_axis."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import assert_close, assert_op_close, bitwise_equal, to_np
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu
OPS = ["mean", "max", "min", "norm"]


def check_axis(shape, dim, op, dist="normal", seed=5, offset=0):
    x = inputs.make(shape, dist, seed)
    o, r, i = L.canonical_axis(x.shape, dim)
    ref, scale = oracle.reduce_op(x.numpy(), o, r, i, op)
    got = L.reduce_axis_op_f32(on_device(x, offset), dim, op)
    assert_op_close(got, ref, scale, op, r, f"{op} {shape} dim={dim} off={offset}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("n", [1, 3, 1000, 8193, 1_000_003, 50_000_000])
@pytest.mark.parametrize("offset", [0, 1])
def test_1d(op, n, offset):
    x = inputs.make((n,), "uniform_pm1", 40 + n % 7)
    ref, scale = oracle.reduce_op(x.numpy(), 1, n, 1, op)
    got = L.reduce_f32(on_device(x, offset), op)
    assert_op_close(got, ref, scale, op, n, f"{op} n={n} off={offset}")


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("shape,dim", [((64, 1000), 1), ((300, 2049), 1), ((70, 65536), 1), ((5, 300001), 1),
                                       ((128, 512, 257), 1), ((4, 3000, 4096), 1), ((65536, 64), 0),
                                       ((2, 777, 4095), 1), ((6, 5, 4, 3), 2)])
def test_axis(op, shape, dim):
    check_axis(shape, dim, op)


@pytest.mark.parametrize("op", OPS)
def test_axis_split_and_misaligned(op):
    check_axis((1, 65536, 1024), 1, op)     # split reduce axis, last-block combine
    check_axis((3, 2000, 36), 1, op, offset=1)  # scalar columns on a misaligned base


@pytest.mark.parametrize("op", ["max", "min"])
def test_nan_propagates(op):
    x = inputs.make((4, 5000), "uniform01", 2)
    x[2, 4321] = float("nan")
    got = L.reduce_axis_op_f32(on_device(x), 1, op).cpu().numpy()
    assert np.isnan(got[2]) and np.isfinite(np.delete(got, 2)).all()
    y = inputs.make((3_000_000,), "uniform01", 2)
    y[1_234_567] = float("nan")
    assert math.isnan(L.reduce_f32(on_device(y), op).item())


def test_empty_values():
    x = torch.empty((3, 0, 2), device="cuda")
    want = {"sum": 0.0, "mean": float("nan"), "max": -float("inf"), "min": float("inf"), "norm": 0.0}
    for op, v in want.items():
        got = L.reduce_axis_op_f32(x, 1, op).cpu().numpy()
        if math.isnan(v):
            assert np.isnan(got).all(), op
        else:
            assert (got == v).all(), op


def test_integer_inputs():
    x = inputs.make((16, 4096, 36), "int:-8:8", 9)
    for op in ("max", "min"):
        ref, _ = oracle.reduce_op(x.numpy(), 16, 4096, 36, op)
        assert np.array_equal(L.reduce_axis_op_f32(on_device(x), 1, op).cpu().numpy().reshape(-1), ref.reshape(-1))
    xi = x.numpy().astype(np.int64)
    ss = (xi * xi).sum(axis=1).astype(np.float64)  # exact in fp32 as well (< 2^24)
    got = L.reduce_axis_op_f32(on_device(x), 1, "norm").cpu().numpy()
    assert np.array_equal(got, np.sqrt(ss).astype(np.float32))


def test_deterministic_bitwise():
    xd = on_device(inputs.make((4096, 4096), "normal", 1))
    for op in OPS:
        for dim in (0, 1):
            a = L.reduce_axis_op_f32(xd, dim, op).clone()
            b = L.reduce_axis_op_f32(xd, dim, op).clone()
            assert bitwise_equal(a, b), (op, dim)
        a = L.reduce_f32(xd, op).clone()
        assert bitwise_equal(a, L.reduce_f32(xd, op)), op


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("shape", [(3, 5000, 4), (2, 30001, 3), (5, 999, 32), (2, 4000, 128), (64, 100, 6)])
@pytest.mark.parametrize("split", [0, 9])
def test_narrow_rows_ops(op, shape, split):
    """Mean, max, min and norm on the narrow-row kernel, with and without
    forced slices (the last block combines them), and a warp per plane."""
    L.set_option(L.OPT_AXIS_SPLIT, split)
    check_axis(shape, 1, op)
    check_axis(shape, 1, op, offset=1)
    L.set_option(L.OPT_COLS_VARIANT, 7)
    check_axis(shape, 1, op)
    check_axis((3000, 50, shape[2]), 1, op, offset=1)


# Reductions along rows of at most 2048 elements (inner == 1): one warp per
# row (OPT_ROWS_FORM 1) or chunks of whole rows staged in shared memory with a
# group of 1-32 lanes per row (2, the automatic choice).
SHORT_N = [1, 2, 3, 6, 7, 8, 31, 32, 33, 50, 64, 65, 99, 100, 127, 130, 255, 256, 257, 1000, 1024, 2047, 2048]


@pytest.mark.parametrize("op", OPS + ["sum"])
@pytest.mark.parametrize("form", [1, 2])
def test_short_rows_both_forms(op, form):
    L.set_option(L.OPT_ROWS_FORM, form)
    for n in SHORT_N:
        rows = 3 * max(1, 3072 // n) + 5
        for offset in (0, 1):
            x = inputs.make((rows, n), "normal", 50 + n % 11)
            got = L.reduce_axis_op_f32(on_device(x, offset), 1, op)
            what = f"{op} [{rows},{n}] form={form} off={offset}"
            if op == "sum":
                ref, scale = oracle.axis_sum(x.numpy(), rows, n, 1)
                assert_close(to_np(got).reshape(-1), ref.reshape(-1), scale.reshape(-1), what)
            else:
                ref, scale = oracle.reduce_op(x.numpy(), rows, n, 1, op)
                assert_op_close(got, ref, scale, op, n, what)


def test_short_rows_forms_exact_and_deterministic():
    """Small integers sum exactly in both forms (so they agree bit for bit),
    and max / min pick the same elements; reruns are bit-identical."""
    for n in (5, 32, 66, 100, 1000):
        x = on_device(inputs.make((20_000, n), "int:-8:8", 61))
        outs = {}
        for form in (1, 2):
            L.set_option(L.OPT_ROWS_FORM, form)
            for op in ("sum", "max", "min"):
                a = L.reduce_axis_op_f32(x, 1, op)
                assert bitwise_equal(L.reduce_axis_op_f32(x, 1, op), a)
                outs[(form, op)] = a
        for op in ("sum", "max", "min"):
            assert bitwise_equal(outs[(1, op)], outs[(2, op)]), (n, op)
    L.check()
