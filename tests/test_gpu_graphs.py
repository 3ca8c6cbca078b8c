"""Calls captured into a CUDA graph replay correctly (GPU).

After a first call on the device (which allocates the library workspace), the
entry points may be captured: the reductions reset their tickets on the
device, and the look-back scan takes its launch epoch from a device word that
every launch advances, so a replay never mistakes the flags of an earlier
replay for its own.  Each replay runs on new input values and is compared,
bit for bit, with eager calls on the same values."""
import pytest
import torch

from gpu_common import libreduce_defaults, on_device  # noqa: F401
from parity import bitwise_equal
from reduction_scan_primitives_gb300 import inputs
from reduction_scan_primitives_gb300 import libreduce as L

pytestmark = pytest.mark.gpu


def calls(x1, xa, xl, xn, xc, outs, ws):
    L.reduce_sum_f32(x1, out=outs["sum"])
    L.reduce_axis_f32(xa, 1, out=outs["axis"])
    L.reduce_axis_op_f32(xa, 1, "max", out=outs["max"])
    L.reverse_cumsum_f32(xl, out=outs["lookback"])           # few long rows: the look-back scan
    L.cumsum_f32(xl, 1, exclusive=True, out=outs["forward"])  # the look-back, mirrored
    L.cumsum_f32(xn, 1, out=outs["narrow"])                   # narrow rows, segmented
    L.cumsum_f32(xc, 1, reverse=True, out=outs["cols"])       # few column tiles: the column look-back
    L.set_option(L.OPT_AXIS_SPLIT, 6)
    L.cumsum_f32(xc, 1, exclusive=True, out=outs["cols3"])     # the same, forced into three passes
    L.set_option(L.OPT_AXIS_SPLIT, 0)
    L.cumsum_ws_f32(xl, 1, reverse=True, ws=ws, out=outs["lookback_ws"])


def test_capture_and_replay():
    shapes = {"x1": (3_000_001,), "xa": (8, 1000, 300), "xl": (2, 3_000_000), "xn": (1, 400_000, 4),
              "xc": (1, 5000, 4096)}
    xs = {k: on_device(inputs.make(s, "uniform_pm1", 1)) for k, s in shapes.items()}
    outs = {"sum": torch.empty((), device="cuda"), "axis": torch.empty(8, 300, device="cuda"),
            "max": torch.empty(8, 300, device="cuda"), "lookback": torch.empty_like(xs["xl"]),
            "forward": torch.empty_like(xs["xl"]), "narrow": torch.empty_like(xs["xn"]),
            "cols": torch.empty_like(xs["xc"]), "cols3": torch.empty_like(xs["xc"]),
            "lookback_ws": torch.empty_like(xs["xl"])}
    ws = L.workspace(L.cumsum_ws_f32(xs["xl"], 1, reverse=True))
    args = (xs["x1"], xs["xa"], xs["xl"], xs["xn"], xs["xc"], outs, ws)
    calls(*args)  # the first calls allocate the library workspace
    torch.cuda.synchronize()
    L.check()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls(*args)

    for seed in range(2, 7):
        for k, s in shapes.items():  # new values in the captured buffers
            xs[k].copy_(inputs.make(s, "uniform_pm1", seed).to("cuda"))
        graph.replay()
        torch.cuda.synchronize()
        L.check()
        L.check_ws(ws)
        got = {k: v.clone() for k, v in outs.items()}
        eager = {k: torch.empty_like(v) for k, v in outs.items()}
        calls(xs["x1"], xs["xa"], xs["xl"], xs["xn"], xs["xc"], eager, ws)
        torch.cuda.synchronize()
        L.check()
        for k in outs:
            assert bitwise_equal(got[k], eager[k]), (seed, k)
