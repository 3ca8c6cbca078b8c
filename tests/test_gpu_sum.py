"""reduce_sum_f32 against the oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import assert_close, assert_exact, bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu


def gpu_sum(x_cpu, offset=0):
    return L.reduce_sum_f32(on_device(x_cpu.reshape(-1), offset)).item()


def test_harmonic_1e6():
    """x[i] = 1/(i+1), n = 1e6: the oracle's value and the harmonic number."""
    n = 1_000_000
    x = inputs.make((n,), "harmonic")
    s = gpu_sum(x)
    ref, scale = oracle.sum1d(x.numpy())
    assert_close(s, ref, scale, "harmonic")
    h = pins.harmonic_closed_form(n)
    assert abs(s - h) <= oracle.tolerance(scale)


def test_uniform_pm1_1e6():
    x = inputs.make((1_000_000,), "uniform_pm1", 42)
    ref, scale = oracle.sum1d(x.numpy())
    assert_close(gpu_sum(x), ref, scale, "uniform[-1,1) n=1e6")


EDGE_N = [0, 1, 2, 3, 4, 5, 31, 32, 33, 255, 256, 257, 1023, 1024, 1025, 8191, 8192, 8193,
          65537, 1_000_003, 2 ** 24 - 1, 2 ** 24, 2 ** 24 + 1]


@pytest.mark.parametrize("n", EDGE_N)
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_edge_sizes_and_alignment(n, offset):
    x = inputs.make((n,), "uniform_pm1", 1000 + n % 97)
    ref, scale = oracle.sum1d(x.numpy())
    s = gpu_sum(x, offset)
    if n == 0:
        assert s == 0.0
    assert_close(s, ref, scale, f"n={n} offset={offset}")


@pytest.mark.parametrize("dist,n", [("int:-1:1", 1_000_000), ("int:-1:1", 10_000_000),
                                    ("int:-8:8", 1_000_000), ("int:0:3", 4_000_000)])
def test_integer_inputs_exact(dist, n):
    x = inputs.make((n,), dist, 42)
    ref, _ = oracle.sum1d(x.numpy())
    assert_exact(gpu_sum(x), ref, dist)
    assert_exact(gpu_sum(x, 3), ref, dist + " misaligned")


@pytest.mark.parametrize("n", [10_000, 100_000, 1_000_000, 10_000_000, 100_000_000])
def test_sweep_uniform01(n):
    x = inputs.make((n,), "uniform01", 42)
    ref, scale = oracle.sum1d(x.numpy())
    assert_close(gpu_sum(x), ref, scale, f"sweep n={n}")


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("waves", [1, 3])
def test_launch_variants(variant, waves):
    x = inputs.make((3_000_017,), "normal", 5)
    ref, scale = oracle.sum1d(x.numpy())
    L.set_option(L.OPT_CONTIG_VARIANT, variant)
    L.set_option(L.OPT_WAVES, waves)
    assert_close(gpu_sum(x, 1), ref, scale, f"variant {variant} waves {waves}")


@pytest.mark.parametrize("chunks", [1, 2, 7, 1000])
def test_forced_chunks(chunks):
    x = inputs.make((2_000_001,), "uniform_pm1", 8)
    ref, scale = oracle.sum1d(x.numpy())
    L.set_option(L.OPT_AXIS_SPLIT, chunks)
    assert_close(gpu_sum(x, 2), ref, scale, f"chunks {chunks}")


def test_deterministic_bitwise():
    x = on_device(inputs.make((10_000_000,), "uniform_pm1", 9))
    outs = [L.reduce_sum_f32(x).clone() for _ in range(3)]
    for o in outs[1:]:
        assert bitwise_equal(outs[0], o)


def test_nan_and_inf_propagate():
    x = inputs.make((100_000,), "uniform01", 1)
    x[777] = float("nan")
    assert np.isnan(gpu_sum(x))
    x = inputs.make((100_000,), "uniform01", 1)
    x[5] = float("inf")
    assert gpu_sum(x) == float("inf")
    x[6] = float("-inf")
    assert np.isnan(gpu_sum(x))


def test_out_tensor_and_stream():
    x = on_device(inputs.make((123_457,), "uniform_pm1", 2))
    out = torch.full((1,), 7.0, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        L.reduce_sum_f32(x, out=out)
    torch.cuda.current_stream().wait_stream(s)
    ref, scale = oracle.sum1d(x.cpu().numpy())
    assert_close(out.item(), ref, scale, "side stream")
