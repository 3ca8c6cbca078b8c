"""The C ABI from C: a C99 program built against include/libreduce.h alone
(warnings as errors, no CUDA header) links with libreduce and gets the
documented statuses for calls decided before any CUDA work.  CPU only."""
import os
import shutil
import subprocess

import pytest

from reduction_scan_primitives_gb300 import build as lib_build
from reduction_scan_primitives_gb300 import libreduce as L

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def caller(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lib_build.build()
    exe = str(tmp_path_factory.mktemp("c") / "caller")
    libdir = os.path.dirname(L.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "c", "caller.c"),
                    "-L", libdir, "-lreduce", f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    return dict(line.split(" ", 1) for line in out.splitlines())


def test_statuses_from_c(caller):
    expect = {"sum_negative_n": L.ERR_INVALID_ARG, "sum_null_x": L.ERR_INVALID_ARG,
              "sum_overflow": L.ERR_OVERFLOW, "axis_negative": L.ERR_INVALID_ARG,
              "op_unknown": L.ERR_INVALID_ARG, "scan_bad_flags": L.ERR_INVALID_ARG,
              "scan_alias": L.ERR_ALIAS, "scan_empty": L.OK, "ws_query_empty": L.OK,
              "ws_query_bytes": 0, "ws_null_size": L.ERR_INVALID_ARG,
              "option_unknown": L.ERR_INVALID_ARG, "option_default": L.OK}
    got = {k: int(caller[k]) for k in expect}
    assert got == expect
    assert caller["strerror_alias"] == "output overlaps input"
    assert int(caller["launches"]) == 0
