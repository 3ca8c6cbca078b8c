"""The debug build (build(debug=True) -> libreduce_debug.so): it builds
without a GPU, exports the same C ABI as the release library, and says which
it is; its calls decide the same statuses before any device work."""
import ctypes

import pytest

from reduction_scan_primitives_gb300 import build as lib_build
from reduction_scan_primitives_gb300 import libreduce as L


@pytest.fixture(scope="module")
def dbg():
    path = lib_build.build(debug=True)
    lib = L.load(path)
    return lib


def test_same_entry_points(dbg):
    for name in L.declared_functions():
        assert hasattr(dbg, name), name


def test_reports_its_build(dbg):
    assert dbg.libreduce_debug_build() == 1
    assert L.load().libreduce_debug_build() == 0
    assert dbg.libreduce_debug_bad_address() == 0


def test_statuses_before_device_work(dbg):
    vp = ctypes.c_void_p
    assert dbg.reduce_sum_f32(None, -1, vp(16), None) == L.ERR_INVALID_ARG
    assert dbg.cumsum_f32(vp(16), 1, 4, 1, vp(16), 8, None) == L.ERR_INVALID_ARG
    assert dbg.reduce_axis_f32(vp(16), 1 << 62, 1 << 62, 1, vp(32), None) == L.ERR_OVERFLOW
    assert dbg.libreduce_strerror(L.ERR_BOUNDS).startswith(b"debug build")
