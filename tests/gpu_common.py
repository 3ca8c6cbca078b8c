"""Shared fixtures for the GPU parity tests."""
import pytest
import torch

from reduction_scan_primitives_gb300 import build as lib_build
from reduction_scan_primitives_gb300 import libreduce as L

DEFAULT_OPTIONS = ((L.OPT_SCAN_STRATEGY, 0), (L.OPT_AXIS_SPLIT, 0), (L.OPT_SPIN_LIMIT, 0),
                   (L.OPT_STALL_TILE, -1), (L.OPT_CONTIG_VARIANT, -1), (L.OPT_COLS_VARIANT, -1),
                   (L.OPT_RSCAN_VARIANT, -1), (L.OPT_WAVES, 0), (L.OPT_LOOKBACK_LAG, 0),
                   (L.OPT_SCAN_COLS_VARIANT, -1), (L.OPT_ROWS_FORM, 0))


def reset_options():
    for opt, val in DEFAULT_OPTIONS:
        L.set_option(opt, val)


@pytest.fixture(autouse=True)
def libreduce_defaults():
    lib_build.build()
    L.load()
    reset_options()
    yield
    reset_options()
    L.check()


def on_device(x_cpu, offset=0):
    """Copy x to the GPU at a chosen 4-byte offset from a fresh allocation."""
    n = x_cpu.numel()
    buf = torch.empty(n + 8, dtype=torch.float32, device="cuda")
    xd = buf[offset:offset + n].view(x_cpu.shape)
    xd.copy_(x_cpu)
    return xd
