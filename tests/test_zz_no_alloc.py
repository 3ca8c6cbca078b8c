"""reduce_sum_f32_noalloc, the 1D sum that allocates nothing (GPU).

Callers that cannot allocate device memory (inside a custom allocator, a
memory-capped service, a stream capture) use this entry point: its scratch is
a fixed static device array instead of the library's cudaMalloc'd workspace.
Here it is called through the C ABI and checked against reduce_sum_f32 on two
calls in a row (the array keeps the previous call's contents, so the second
call shows that what must start at zero is cleared).  This file is collected
last; it passes both alone in a fresh process and after the other tests.
"""
import ctypes

import pytest
import torch

import oracle
from reduction_scan_primitives_gb300 import build as lib_build
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return L.load()


def _call(lib, x, out):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.reduce_sum_f32_noalloc(ctypes.c_void_p(x.data_ptr()), x.numel(),
                                      ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream))


@pytest.mark.parametrize("n", [1, 1000, 1_000_003, 50_000_001, 300_000_000])
def test_matches_reduce_sum_on_two_calls(lib, n):
    x = inputs.make((n,), "uniform_pm1", 17, device="cuda")
    ref = torch.empty((), device="cuda")
    assert lib.reduce_sum_f32(ctypes.c_void_p(x.data_ptr()), n, ctypes.c_void_p(ref.data_ptr()),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == L.OK
    _, scale = oracle.sum1d(x.cpu().numpy())
    tol = float(oracle.tolerance(scale))
    for _ in range(2):
        out = torch.full((), float("nan"), device="cuda")
        assert _call(lib, x, out) == L.OK
        torch.cuda.synchronize()
        assert abs(out.item() - ref.item()) <= tol, (n, out.item(), ref.item(), tol)


def test_empty_and_limits(lib):
    out = torch.full((), 5.0, device="cuda")
    x = torch.empty(0, device="cuda")
    assert _call(lib, x, out) == L.OK
    torch.cuda.synchronize()
    assert out.item() == 0.0
    # Beyond the stated maximum (2^36 floats): rejected on the host.
    x1 = torch.zeros(1, device="cuda")
    assert lib.reduce_sum_f32_noalloc(ctypes.c_void_p(x1.data_ptr()), (1 << 36) + 1,
                                      ctypes.c_void_p(out.data_ptr()), None) == L.ERR_OVERFLOW
    assert lib.reduce_sum_f32_noalloc(None, 5, ctypes.c_void_p(out.data_ptr()), None) == L.ERR_INVALID_ARG


def test_python_binding_matches(lib):
    x = inputs.make((2_000_003,), "uniform_pm1", 19, device="cuda")
    a = L.reduce_sum_f32_noalloc(x).clone()
    b = L.reduce_sum_f32(x)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
