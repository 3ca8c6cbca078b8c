"""The all-core CPU baseline of the benchmark (threaded.c): the three
primitives in fp64 on every core the process may run on, fp32 in and fp32 out.

A reported context number for bench.py, nothing more: the parity reference is
the single-threaded oracle, and neither the library nor its tests use this.
"""
import ctypes
import os
import platform
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "threaded.c")
LIB = os.path.join(HERE, "libcpubase.so")

_lib = None
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O3", "-std=c99", "-fPIC", "-shared", "-pthread", "-Wall", "-o", tmp, SRC],
                       check=True)
        os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.cpub_sum.argtypes = [_f32p, i64, i32, _f32p]
        lib.cpub_axis_sum.argtypes = [_f32p, i64, i64, i64, i32, _f32p]
        lib.cpub_reverse_cumsum.argtypes = [_f32p, i64, i64, i32, _f32p]
        for f in (lib.cpub_sum, lib.cpub_axis_sum, lib.cpub_reverse_cumsum):
            f.restype = i32
        _lib = lib
    return _lib


def cores() -> int:
    return len(os.sched_getaffinity(0))


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def _check(rc):
    if rc != 0:
        raise RuntimeError("cpu baseline failed")


def sum1d(x, threads=None):
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(1, np.float32)
    _check(_load().cpub_sum(x, x.size, threads or cores(), out))
    return float(out[0])


def axis_sum(x, outer, reduce, inner, threads=None):
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(outer * inner, np.float32)
    _check(_load().cpub_axis_sum(x, outer, reduce, inner, threads or cores(), out))
    return out.reshape(outer, inner)


def reverse_cumsum(x, rows, N, threads=None):
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    y = np.empty(rows * N, np.float32)
    _check(_load().cpub_reverse_cumsum(x, rows, N, threads or cores(), y))
    return y.reshape(rows, N)
