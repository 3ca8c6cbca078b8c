"""Thin ctypes binding of libreduce (include/libreduce.h).

Argument marshalling only: every value is computed by the CUDA kernels behind
the C ABI.  There is no fallback: if libreduce.so is missing or the tensor is
not a contiguous float32 CUDA tensor, the call raises.

The functions carry the C entry points' names and take torch tensors; the
work is queued on the current torch stream of the tensor's device.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import re

import torch

from . import build as _build

OK = 0
ERR_INVALID_ARG = 1
ERR_OVERFLOW = 2
ERR_ALIAS = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_BOUNDS = 6  # debug build only: a kernel access outside its call's buffers was skipped

OPS = {"sum": 0, "mean": 1, "max": 2, "min": 3, "norm": 4}

SCAN_REVERSE = 1
SCAN_EXCLUSIVE = 2

OPT_SCAN_STRATEGY = 1
OPT_AXIS_SPLIT = 2
OPT_SPIN_LIMIT = 3
OPT_STALL_TILE = 4
OPT_CONTIG_VARIANT = 5
OPT_COLS_VARIANT = 6
OPT_RSCAN_VARIANT = 7
OPT_WAVES = 8
OPT_LOOKBACK_LAG = 9
OPT_SCAN_COLS_VARIANT = 10
OPT_ROWS_FORM = 11

# The library this binding loads: the release build, or another build of the
# same C ABI named by LIBREDUCE_LIB (e.g. the debug build, _build.DEBUG_LIB).
LIB_PATH = os.environ.get("LIBREDUCE_LIB") or _build.LIB
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "libreduce.h")

_lib = None


class LibreduceError(RuntimeError):
    """A libreduce call returned a nonzero status."""

    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{fn} failed: status {status}"
        if _lib is not None:
            msg += f" ({_lib.libreduce_strerror(status).decode()})"
        if status == ERR_CUDA:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


def declared_functions() -> list[str]:
    """Names of the functions include/libreduce.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:LIBREDUCE_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*"
                      r"([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libreduce.so (built in-tree by reduction_scan_primitives_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libreduce is not built ({p} is missing); run reduction_scan_primitives_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.reduce_sum_f32.argtypes = [vp, i64, vp, vp]
    lib.reduce_sum_f32.restype = i32
    lib.reduce_sum_f32_noalloc.argtypes = [vp, i64, vp, vp]
    lib.reduce_sum_f32_noalloc.restype = i32
    lib.reduce_axis_f32.argtypes = [vp, i64, i64, i64, vp, vp]
    lib.reduce_axis_f32.restype = i32
    lib.reduce_f32.argtypes = [vp, i64, vp, i32, vp]
    lib.reduce_f32.restype = i32
    lib.reduce_axis_op_f32.argtypes = [vp, i64, i64, i64, vp, i32, vp]
    lib.reduce_axis_op_f32.restype = i32
    lib.reverse_cumsum_f32.argtypes = [vp, i64, i64, vp, vp]
    lib.reverse_cumsum_f32.restype = i32
    lib.cumsum_f32.argtypes = [vp, i64, i64, i64, vp, ctypes.c_uint, vp]
    lib.cumsum_f32.restype = i32
    lib.libreduce_check.argtypes = [vp]
    lib.libreduce_check.restype = i32
    sz = ctypes.POINTER(ctypes.c_size_t)
    lib.reduce_axis_op_ws_f32.argtypes = [vp, i64, i64, i64, vp, i32, vp, sz, vp]
    lib.reduce_axis_op_ws_f32.restype = i32
    lib.cumsum_ws_f32.argtypes = [vp, i64, i64, i64, vp, ctypes.c_uint, vp, sz, vp]
    lib.cumsum_ws_f32.restype = i32
    lib.libreduce_check_ws.argtypes = [vp, vp]
    lib.libreduce_check_ws.restype = i32
    lib.libreduce_strerror.argtypes = [i32]
    lib.libreduce_strerror.restype = ctypes.c_char_p
    lib.libreduce_last_cuda_error.argtypes = []
    lib.libreduce_last_cuda_error.restype = i32
    lib.libreduce_launch_count.argtypes = []
    lib.libreduce_launch_count.restype = i64
    lib.libreduce_set_option.argtypes = [i32, i64]
    lib.libreduce_set_option.restype = i32
    lib.libreduce_debug_build.argtypes = []
    lib.libreduce_debug_build.restype = i32
    lib.libreduce_debug_bad_address.argtypes = []
    lib.libreduce_debug_bad_address.restype = ctypes.c_uint64
    if path is None:
        _lib = lib
    return lib


def _raise_on(fn: str, status: int):
    if status != OK:
        raise LibreduceError(fn, status, _lib.libreduce_last_cuda_error() if _lib else 0)


def _check_tensor(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device}); libreduce has no CPU path")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32 (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# The current stream's raw handle without building a Stream object (the
# public route costs about a microsecond per call).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(device) -> int:
    index = device.index if device.index is not None else torch.cuda.current_device()
    if _raw_stream is not None:
        return _raw_stream(index)
    return torch.cuda.current_stream(index).cuda_stream


def _on(device):
    """Make `device` current for the call, entering it only when it is not."""
    if device.index is None or device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def canonical_axis(shape, dim: int):
    """(outer, reduce, inner) of a contiguous tensor of `shape` reduced along `dim`."""
    nd = len(shape)
    if nd == 0:
        return 1, 1, 1
    if not -nd <= dim < nd:
        raise IndexError(f"dim {dim} out of range for {nd} dims")
    dim %= nd
    outer = 1
    for s in shape[:dim]:
        outer *= int(s)
    inner = 1
    for s in shape[dim + 1:]:
        inner *= int(s)
    return outer, int(shape[dim]), inner


def reduce_sum_f32(x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Sum of every element of x (float32 CUDA, contiguous) -> 0-d float32 tensor."""
    _check_tensor(x, "x")
    if out is None:
        out = torch.empty((), dtype=torch.float32, device=x.device)
    else:
        _check_tensor(out, "out")
        if out.numel() != 1 or out.device != x.device:
            raise ValueError("out must hold one float on x's device")
    lib = load()
    with _on(x.device):
        st = lib.reduce_sum_f32(x.data_ptr(), x.numel(), out.data_ptr(), _stream_ptr(x.device))
    _raise_on("reduce_sum_f32", st)
    return out


def reduce_sum_f32_noalloc(x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """reduce_sum_f32 that allocates no device memory: its scratch is a fixed
    static device array (n <= 2**36; calls must not overlap on the GPU)."""
    _check_tensor(x, "x")
    if out is None:
        out = torch.empty((), dtype=torch.float32, device=x.device)
    else:
        _check_tensor(out, "out")
        if out.numel() != 1 or out.device != x.device:
            raise ValueError("out must hold one float on x's device")
    lib = load()
    with _on(x.device):
        st = lib.reduce_sum_f32_noalloc(x.data_ptr(), x.numel(), out.data_ptr(), _stream_ptr(x.device))
    _raise_on("reduce_sum_f32_noalloc", st)
    return out


def reduce_axis_f32(x: torch.Tensor, dim: int, keepdim: bool = False,
                    out: torch.Tensor | None = None) -> torch.Tensor:
    """Sum of x along `dim` (float32 CUDA, contiguous)."""
    _check_tensor(x, "x")
    outer, reduce, inner = canonical_axis(x.shape, dim)
    shape = list(x.shape)
    d = dim % x.dim() if x.dim() else 0
    if x.dim():
        if keepdim:
            shape[d] = 1
        else:
            del shape[d]
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=x.device)
    else:
        _check_tensor(out, "out")
        if out.numel() != outer * inner or out.device != x.device:
            raise ValueError("out has the wrong size or device")
    lib = load()
    with _on(x.device):
        st = lib.reduce_axis_f32(x.data_ptr(), outer, reduce, inner, out.data_ptr(),
                                 _stream_ptr(x.device))
    _raise_on("reduce_axis_f32", st)
    return out


def _op_code(op) -> int:
    if isinstance(op, str):
        if op not in OPS:
            raise ValueError(f"unknown reduction {op!r}; one of {sorted(OPS)}")
        return OPS[op]
    return int(op)


def reduce_f32(x: torch.Tensor, op="sum", out: torch.Tensor | None = None) -> torch.Tensor:
    """Reduction of every element of x: "sum", "mean", "max", "min" or "norm"."""
    _check_tensor(x, "x")
    if out is None:
        out = torch.empty((), dtype=torch.float32, device=x.device)
    else:
        _check_tensor(out, "out")
        if out.numel() != 1 or out.device != x.device:
            raise ValueError("out must hold one float on x's device")
    lib = load()
    with _on(x.device):
        st = lib.reduce_f32(x.data_ptr(), x.numel(), out.data_ptr(), _op_code(op), _stream_ptr(x.device))
    _raise_on("reduce_f32", st)
    return out


def reduce_axis_op_f32(x: torch.Tensor, dim: int, op="sum", keepdim: bool = False,
                       out: torch.Tensor | None = None) -> torch.Tensor:
    """Reduction of x along `dim`: "sum", "mean", "max", "min" or "norm"."""
    _check_tensor(x, "x")
    outer, reduce, inner = canonical_axis(x.shape, dim)
    shape = list(x.shape)
    if x.dim():
        d = dim % x.dim()
        if keepdim:
            shape[d] = 1
        else:
            del shape[d]
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=x.device)
    else:
        _check_tensor(out, "out")
        if out.numel() != outer * inner or out.device != x.device:
            raise ValueError("out has the wrong size or device")
    lib = load()
    with _on(x.device):
        st = lib.reduce_axis_op_f32(x.data_ptr(), outer, reduce, inner, out.data_ptr(), _op_code(op),
                                    _stream_ptr(x.device))
    _raise_on("reduce_axis_op_f32", st)
    return out


def reverse_cumsum_f32(x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """y[..., j] = sum over k >= j of x[..., k] along the last dim (float32 CUDA)."""
    _check_tensor(x, "x")
    if x.dim() == 0:
        raise ValueError("x must have at least one dim")
    N = int(x.shape[-1])
    rows = x.numel() // N if N else 0
    if out is None:
        out = torch.empty_like(x)
    else:
        _check_tensor(out, "out")
        if out.shape != x.shape or out.device != x.device:
            raise ValueError("out must have x's shape and device")
    lib = load()
    with _on(x.device):
        st = lib.reverse_cumsum_f32(x.data_ptr(), rows, N, out.data_ptr(), _stream_ptr(x.device))
    _raise_on("reverse_cumsum_f32", st)
    return out


def cumsum_f32(x: torch.Tensor, dim: int = -1, reverse: bool = False, exclusive: bool = False,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """Cumulative sum of x along `dim` (float32 CUDA, contiguous): forward
    (sum over k <= j) or reverse (k >= j), inclusive or exclusive (k != j)."""
    _check_tensor(x, "x")
    if x.dim() == 0:
        raise ValueError("x must have at least one dim")
    outer, N, inner = canonical_axis(x.shape, dim)
    if out is None:
        out = torch.empty_like(x)
    else:
        _check_tensor(out, "out")
        if out.shape != x.shape or out.device != x.device:
            raise ValueError("out must have x's shape and device")
    flags = (SCAN_REVERSE if reverse else 0) | (SCAN_EXCLUSIVE if exclusive else 0)
    lib = load()
    with _on(x.device):
        st = lib.cumsum_f32(x.data_ptr(), outer, N, inner, out.data_ptr(), flags, _stream_ptr(x.device))
    _raise_on("cumsum_f32", st)
    return out


def _ws_ptr(ws, device=None):
    if ws is None:
        return None
    if not isinstance(ws, torch.Tensor) or ws.device.type != "cuda":
        raise ValueError("the workspace must be a CUDA tensor")
    if device is not None and ws.device != device:
        raise ValueError("the workspace must be on x's device")
    if not ws.is_contiguous():
        raise ValueError("the workspace must be contiguous")
    return ws.data_ptr()


def _ws_nbytes(ws):
    return ctypes.c_size_t(0 if ws is None else ws.numel() * ws.element_size())


def reduce_axis_op_ws_f32(x: torch.Tensor, dim: int, op="sum", ws: torch.Tensor | None = None,
                          out: torch.Tensor | None = None):
    """reduce_axis_op_f32 with caller scratch.  ws=None: returns the bytes the
    call needs (nothing runs); else runs with `ws` (a 256-byte aligned CUDA
    buffer of at least that many bytes) and returns the output."""
    _check_tensor(x, "x")
    outer, reduce, inner = canonical_axis(x.shape, dim)
    if out is None:
        shape = list(x.shape)
        if x.dim():
            del shape[dim % x.dim()]
        out = torch.empty(shape, dtype=torch.float32, device=x.device)
    else:
        _check_tensor(out, "out")
        if out.numel() != outer * inner or out.device != x.device:
            raise ValueError("out has the wrong size or device")
    nbytes = _ws_nbytes(ws)
    lib = load()
    with _on(x.device):
        st = lib.reduce_axis_op_ws_f32(x.data_ptr(), outer, reduce, inner, out.data_ptr(), _op_code(op),
                                       _ws_ptr(ws, x.device), ctypes.byref(nbytes), _stream_ptr(x.device))
    _raise_on("reduce_axis_op_ws_f32", st)
    return int(nbytes.value) if ws is None else out


def cumsum_ws_f32(x: torch.Tensor, dim: int = -1, reverse: bool = False, exclusive: bool = False,
                  ws: torch.Tensor | None = None, out: torch.Tensor | None = None):
    """cumsum_f32 with caller scratch (see reduce_axis_op_ws_f32)."""
    _check_tensor(x, "x")
    if x.dim() == 0:
        raise ValueError("x must have at least one dim")
    outer, N, inner = canonical_axis(x.shape, dim)
    if out is None:
        out = torch.empty_like(x)
    else:
        _check_tensor(out, "out")
        if out.shape != x.shape or out.device != x.device:
            raise ValueError("out must have x's shape and device")
    flags = (SCAN_REVERSE if reverse else 0) | (SCAN_EXCLUSIVE if exclusive else 0)
    nbytes = _ws_nbytes(ws)
    lib = load()
    with _on(x.device):
        st = lib.cumsum_ws_f32(x.data_ptr(), outer, N, inner, out.data_ptr(), flags, _ws_ptr(ws, x.device),
                               ctypes.byref(nbytes), _stream_ptr(x.device))
    _raise_on("cumsum_ws_f32", st)
    return int(nbytes.value) if ws is None else out


def check_ws(ws: torch.Tensor) -> None:
    """Synchronise the current stream and raise if a wait of a workspace call ran out."""
    with _on(ws.device):
        st = load().libreduce_check_ws(ws.data_ptr(), _stream_ptr(ws.device))
    _raise_on("libreduce_check_ws", st)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned uint8 CUDA buffer of at least `nbytes` bytes."""
    n = max(int(nbytes), 1)
    raw = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % 256
    return raw[off:off + n]


def check(device=None) -> None:
    """Synchronise the current stream and raise if a device-side wait ran out."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = lib.libreduce_check(_stream_ptr(dev))
    _raise_on("libreduce_check", st)


def set_option(option: int, value: int) -> None:
    _raise_on("libreduce_set_option", load().libreduce_set_option(option, value))


def launch_count() -> int:
    return int(load().libreduce_launch_count())


def debug_build() -> bool:
    """True when the loaded library is the debug build (checked kernel accesses)."""
    return bool(load().libreduce_debug_build())


def debug_bad_address() -> int:
    """The first bad address the last ERR_BOUNDS report found (0: none)."""
    return int(load().libreduce_debug_bad_address())


# Short aliases.
reduce_sum = reduce_sum_f32
reduce_axis = reduce_axis_f32
reverse_cumsum = reverse_cumsum_f32
cumsum = cumsum_f32
