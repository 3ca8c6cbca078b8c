"""reduce_axis_f32 against the oracle (GPU)."""
import itertools

import numpy as np
import pytest

import oracle
from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import assert_close, assert_exact, bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu


def gpu_axis(x_cpu, outer, reduce, inner, offset=0):
    xd = on_device(x_cpu.reshape(outer, reduce, inner), offset)
    return L.reduce_axis_f32(xd, 1).cpu().numpy().reshape(outer, inner)


def check(outer, reduce, inner, dist="normal", seed=3, offset=0, what=""):
    x = inputs.make((outer, reduce, inner), dist, seed)
    ref, scale = oracle.axis_sum(x.numpy(), outer, reduce, inner)
    got = gpu_axis(x, outer, reduce, inner, offset)
    assert_close(got, ref, scale, what or f"[{outer},{reduce},{inner}] off={offset}")
    return got, ref


INNER = [1, 2, 3, 4, 5, 31, 32, 33, 4095, 4096]
REDUCE = [0, 1, 2, 3, 4097]
OUTER = [1, 2, 128]
GRID = [(o, r, i) for o, r, i in itertools.product(OUTER, REDUCE, INNER) if o * r * i <= 2 ** 22]


@pytest.mark.parametrize("outer,reduce,inner", GRID)
def test_shape_grid(outer, reduce, inner):
    check(outer, reduce, inner)


@pytest.mark.parametrize("outer,reduce,inner", [(3, 257, 4096), (2, 1000, 1024), (5, 77, 36)])
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_input(outer, reduce, inner, offset):
    check(outer, reduce, inner, offset=offset)


@pytest.mark.parametrize("variant", range(6))
@pytest.mark.parametrize("shape", [(3, 1000, 4096), (2, 777, 4095), (1, 5000, 260), (7, 33, 100)])
def test_cols_variants(variant, shape):
    L.set_option(L.OPT_COLS_VARIANT, variant)
    check(*shape, what=f"variant {variant} {shape}")


@pytest.mark.parametrize("split", [1, 2, 3, 7, 64])
@pytest.mark.parametrize("shape", [(1, 6000, 4096), (2, 1001, 4095), (4, 20000, 1), (1, 100003, 1)])
def test_forced_split(split, shape):
    L.set_option(L.OPT_AXIS_SPLIT, split)
    check(*shape, dist="uniform_pm1", what=f"split {split} {shape}")


@pytest.mark.parametrize("rows,length", [(1, 1), (3, 1), (1000, 7), (4097, 64), (512, 2048),
                                         (300, 2049), (64, 65536), (5, 300001)])
def test_rows_inner1(rows, length):
    check(rows, length, 1, dist="uniform_pm1")


def test_rows_inner1_misaligned():
    check(513, 1027, 1, offset=1)
    check(70, 9001, 1, offset=3)


@pytest.mark.parametrize("shape", [(3, 500, 77), (64, 4096, 1), (1, 65536, 64), (2, 4096, 4095)])
def test_integer_inputs_exact(shape):
    x = inputs.make(shape, "int:-8:8", 11)
    ref, _ = oracle.axis_sum(x.numpy(), *shape)
    assert_exact(gpu_axis(x, *shape), ref, f"int {shape}")


def test_deterministic_bitwise():
    for shape in [(1, 65536, 512), (128, 4096, 63), (4096, 4096, 1)]:
        L.set_option(L.OPT_AXIS_SPLIT, 0)
        xd = on_device(inputs.make(shape, "uniform_pm1", 4))
        outs = [L.reduce_axis_f32(xd, 1).clone() for _ in range(3)]
        for o in outs[1:]:
            assert bitwise_equal(outs[0], o), shape


def test_zero_reduce_writes_zeros_and_empty_is_noop():
    import torch
    x = torch.empty((4, 0, 5), device="cuda")
    out = L.reduce_axis_f32(x, 1)
    assert out.shape == (4, 5) and bool((out == 0).all())
    x = torch.empty((0, 3, 5), device="cuda")
    assert L.reduce_axis_f32(x, 1).shape == (0, 5)


def test_keepdim_and_dims():
    x = inputs.make((6, 5, 4, 3), "normal", 2)
    xd = on_device(x)
    for dim in range(4):
        o, r, i = L.canonical_axis(x.shape, dim)
        got = L.reduce_axis_f32(xd, dim, keepdim=True)
        shp = list(x.shape)
        shp[dim] = 1
        assert list(got.shape) == shp
        ref, scale = oracle.axis_sum(x.numpy(), o, r, i)
        assert_close(got.cpu().numpy(), ref, scale, f"dim {dim}")


def test_nan_inf():
    x = inputs.make((4, 100, 8), "uniform01", 1)
    x[1, 50, 3] = float("nan")
    x[2, 10, 4] = float("inf")
    got = gpu_axis(x, 4, 100, 8)
    assert np.isnan(got[1, 3]) and got[2, 4] == float("inf")
    assert np.isfinite(np.delete(got.reshape(-1), [1 * 8 + 3, 2 * 8 + 4])).all()


NARROW = [(2, 30000, 4), (5, 777, 3), (3, 1000, 32), (2, 5000, 128), (4, 1001, 12), (1, 200000, 2),
          (100, 300, 7), (2, 70001, 16), (64, 64, 5), (1, 100000, 33), (3, 2000, 100), (2, 3000, 255)]


@pytest.mark.parametrize("shape", NARROW)
@pytest.mark.parametrize("split", [0, 1, 5, 333])
def test_narrow_rows(shape, split):
    """Rows of at most 32 column groups take the narrow kernel (the plane read
    contiguously, a fixed column group per thread, row groups joined by a
    tree), one block per plane or sliced (forced or automatic); the wide
    kernel forced on the same shapes agrees with the oracle too."""
    L.set_option(L.OPT_AXIS_SPLIT, split)
    check(*shape, what=f"narrow {shape} split={split}")
    L.set_option(L.OPT_COLS_VARIANT, 7)  # a warp per plane
    check(*shape, what=f"narrow warp {shape}")
    L.set_option(L.OPT_COLS_VARIANT, 1)
    check(*shape, what=f"wide {shape} split={split}")


@pytest.mark.parametrize("shape", [(5000, 100, 3), (20000, 7, 4), (3000, 64, 32), (2000, 33, 128), (4864, 2, 2)])
def test_narrow_many_small_planes(shape):
    """Many small planes take the warp-per-plane form by default."""
    got, ref = check(*shape, what=f"small planes {shape}")
    x = inputs.make(shape, "int:-8:8", 4)
    ref, _ = oracle.axis_sum(x.numpy(), *shape)
    assert_exact(gpu_axis(x, *shape), ref, f"small planes int {shape}")


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_narrow_rows_misaligned(offset):
    for shape in ((3, 5000, 8), (2, 3001, 32), (2, 999, 128)):
        check(*shape, offset=offset, what=f"narrow {shape} off={offset}")


def test_narrow_rows_integer_exact_and_bitwise():
    for shape, split in (((4, 20000, 4), 0), ((3, 7001, 3), 7), ((2, 100003, 16), 0)):
        L.set_option(L.OPT_AXIS_SPLIT, split)
        x = inputs.make(shape, "int:-8:8", 9)
        ref, _ = oracle.axis_sum(x.numpy(), *shape)
        xd = on_device(x)
        a = L.reduce_axis_f32(xd, 1).clone()
        b = L.reduce_axis_f32(xd, 1).clone()
        assert_exact(a.cpu().numpy(), ref, f"narrow int {shape}")
        assert bitwise_equal(a, b)
