"""The C ABI on the host: the library builds and loads, exports every function
include/libreduce.h declares, and rejects bad arguments before any CUDA call.
CPU only (no GPU is needed or touched)."""
import ctypes
import os
import subprocess

import pytest

from reduction_scan_primitives_gb300 import build as lib_build
from reduction_scan_primitives_gb300 import libreduce as L


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return L.load()


def test_exports_every_declared_symbol(lib):
    names = L.declared_functions()
    assert set(names) >= {"reduce_sum_f32", "reduce_axis_f32", "reverse_cumsum_f32",
                          "libreduce_check", "libreduce_strerror"}
    raw = ctypes.CDLL(L.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in libreduce.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_library_targets_sm103a_only(lib):
    assert ["-gencode", "arch=compute_103a,code=sm_103a"] == lib_build.ARCH
    assert "-use_fast_math" not in " ".join(lib_build.NVCC_FLAGS)


def test_no_dependency_on_shared_cudart(lib):
    out = subprocess.run(["ldd", L.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcudart" not in out


NULL = None
FAKE = 1 << 20  # a 16-byte aligned address never dereferenced by these tests


def test_invalid_arguments_rejected_before_cuda(lib):
    E = L.ERR_INVALID_ARG
    assert lib.reduce_sum_f32(FAKE, -1, FAKE, NULL) == E
    assert lib.reduce_sum_f32(NULL, 5, FAKE, NULL) == E
    assert lib.reduce_sum_f32(FAKE, 5, NULL, NULL) == E
    assert lib.reduce_axis_f32(FAKE, -1, 2, 3, FAKE, NULL) == E
    assert lib.reduce_axis_f32(FAKE, 1, -2, 3, FAKE, NULL) == E
    assert lib.reduce_axis_f32(FAKE, 1, 2, -3, FAKE, NULL) == E
    assert lib.reduce_axis_f32(NULL, 1, 2, 3, FAKE, NULL) == E
    assert lib.reduce_axis_f32(FAKE, 1, 2, 3, NULL, NULL) == E
    assert lib.reverse_cumsum_f32(FAKE, -1, 4, FAKE, NULL) == E
    assert lib.reverse_cumsum_f32(FAKE, 1, -4, FAKE, NULL) == E
    assert lib.reverse_cumsum_f32(NULL, 1, 4, FAKE, NULL) == E
    assert lib.reverse_cumsum_f32(FAKE, 1, 4, NULL, NULL) == E


def test_cumsum_arguments(lib):
    E = L.ERR_INVALID_ARG
    assert lib.cumsum_f32(FAKE, 1, 4, 1, FAKE + 4096, 4, NULL) == E  # unknown flag bit
    assert lib.cumsum_f32(FAKE, -1, 4, 1, FAKE + 4096, 0, NULL) == E
    assert lib.cumsum_f32(FAKE, 1, 4, -2, FAKE + 4096, 0, NULL) == E
    assert lib.cumsum_f32(NULL, 1, 4, 2, FAKE + 4096, 0, NULL) == E
    assert lib.cumsum_f32(FAKE, 2, 4, 3, FAKE + 40, 1, NULL) == L.ERR_ALIAS
    assert lib.cumsum_f32(FAKE, 1 << 62, 4, 1 << 62, FAKE, 0, NULL) == L.ERR_OVERFLOW
    assert lib.cumsum_f32(FAKE, 3, 0, 5, FAKE, 3, NULL) == L.OK  # empty: no-op


def test_reduce_op_arguments(lib):
    E = L.ERR_INVALID_ARG
    assert lib.reduce_f32(FAKE, 16, FAKE + 4096, 9, NULL) == E  # unknown op
    assert lib.reduce_f32(FAKE, 16, FAKE + 4096, -1, NULL) == E
    assert lib.reduce_axis_op_f32(FAKE, 2, 3, 4, FAKE + 4096, 5, NULL) == E
    assert lib.reduce_axis_op_f32(FAKE, 2, 3, 4, FAKE + 4, L.OPS["max"], NULL) == L.ERR_ALIAS
    assert lib.reduce_axis_op_f32(FAKE, 0, 3, 4, FAKE, L.OPS["min"], NULL) == L.OK  # nothing to write
    assert lib.reduce_f32(NULL, 3, FAKE, L.OPS["mean"], NULL) == E


def test_workspace_arguments(lib):
    import ctypes as C
    n = C.c_size_t(1 << 20)
    E = L.ERR_INVALID_ARG
    # ws_bytes NULL, misaligned workspace: rejected before any CUDA call.
    assert lib.reduce_axis_op_ws_f32(FAKE, 1, 8, 1, FAKE + 4096, 0, FAKE + 8192, None, NULL) == E
    assert lib.cumsum_ws_f32(FAKE, 1, 8, 1, FAKE + 4096, 0, FAKE + 8192 + 16, C.byref(n), NULL) == E
    assert lib.reduce_axis_op_ws_f32(FAKE, 1, 8, 1, FAKE + 4096, 0, FAKE + 8192 + 4, C.byref(n), NULL) == E
    # A size query of an empty call needs nothing.
    q = C.c_size_t(77)
    assert lib.cumsum_ws_f32(FAKE, 0, 8, 1, FAKE, 0, NULL, C.byref(q), NULL) == L.OK and q.value == 0
    assert lib.libreduce_check_ws(NULL, NULL) in (E, L.ERR_CUDA)


def test_overflow_rejected(lib):
    big = 1 << 62
    assert lib.reduce_axis_f32(FAKE, big, big, 2, FAKE, NULL) == L.ERR_OVERFLOW
    assert lib.reduce_axis_f32(FAKE, 2, big, 3, FAKE, NULL) == L.ERR_OVERFLOW
    assert lib.reverse_cumsum_f32(FAKE, big, 8, FAKE, NULL) == L.ERR_OVERFLOW
    assert lib.reduce_sum_f32(FAKE, big, FAKE, NULL) == L.ERR_OVERFLOW


def test_alias_rejected(lib):
    assert lib.reverse_cumsum_f32(FAKE, 2, 8, FAKE, NULL) == L.ERR_ALIAS
    assert lib.reverse_cumsum_f32(FAKE, 2, 8, FAKE + 4 * 15, NULL) == L.ERR_ALIAS
    assert lib.reduce_sum_f32(FAKE, 100, FAKE + 40, NULL) == L.ERR_ALIAS
    assert lib.reduce_axis_f32(FAKE, 2, 3, 4, FAKE + 4, NULL) == L.ERR_ALIAS


def test_empty_is_noop_without_cuda(lib):
    # Zero-size outputs need no device: nothing is queued.
    assert lib.reduce_axis_f32(FAKE, 0, 5, 7, FAKE, NULL) == L.OK
    assert lib.reduce_axis_f32(FAKE, 3, 5, 0, FAKE, NULL) == L.OK
    assert lib.reverse_cumsum_f32(FAKE, 0, 5, FAKE, NULL) == L.OK
    assert lib.reverse_cumsum_f32(FAKE, 5, 0, FAKE, NULL) == L.OK


def test_no_cpu_fallback_without_gpu(lib):
    """With valid-looking arguments and no usable GPU, a call reports a CUDA
    error; it never computes anything on the host."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.reduce_sum_f32(FAKE, 16, FAKE + 4096, NULL) == L.ERR_CUDA
    assert lib.libreduce_last_cuda_error() != 0
    with pytest.raises((ValueError, TypeError)):
        L.reduce_sum_f32(torch.ones(8))  # CPU tensor: refused, no fallback


def test_options(lib):
    assert lib.libreduce_set_option(999, 0) == L.ERR_INVALID_ARG
    assert lib.libreduce_set_option(L.OPT_SCAN_STRATEGY, 6) == L.ERR_INVALID_ARG
    assert lib.libreduce_set_option(L.OPT_STALL_TILE, -2) == L.ERR_INVALID_ARG
    for opt, val in ((L.OPT_SCAN_STRATEGY, 0), (L.OPT_AXIS_SPLIT, 0), (L.OPT_SPIN_LIMIT, 0),
                     (L.OPT_STALL_TILE, -1), (L.OPT_CONTIG_VARIANT, -1), (L.OPT_COLS_VARIANT, -1),
                     (L.OPT_RSCAN_VARIANT, -1), (L.OPT_WAVES, 0), (L.OPT_LOOKBACK_LAG, 0),
                     (L.OPT_SCAN_COLS_VARIANT, -1)):
        assert lib.libreduce_set_option(opt, val) == L.OK
    assert lib.libreduce_set_option(L.OPT_SCAN_COLS_VARIANT, 9) == L.OK
    assert lib.libreduce_set_option(L.OPT_SCAN_COLS_VARIANT, 10) == L.ERR_INVALID_ARG
    assert lib.libreduce_set_option(L.OPT_SCAN_COLS_VARIANT, -1) == L.OK
    assert lib.libreduce_set_option(L.OPT_COLS_VARIANT, 9) == L.OK
    assert lib.libreduce_set_option(L.OPT_COLS_VARIANT, 10) == L.ERR_INVALID_ARG
    assert lib.libreduce_set_option(L.OPT_COLS_VARIANT, -1) == L.OK
    for v in (0, 1, 2):
        assert lib.libreduce_set_option(L.OPT_ROWS_FORM, v) == L.OK
    assert lib.libreduce_set_option(L.OPT_ROWS_FORM, 3) == L.ERR_INVALID_ARG
    assert lib.libreduce_set_option(L.OPT_ROWS_FORM, 0) == L.OK


def test_strerror(lib):
    for code in range(6):
        assert lib.libreduce_strerror(code)
    assert lib.libreduce_strerror(77) == b"unknown status"


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        L.load(str(tmp_path / "nope" / "libreduce.so"))


def test_canonical_axis():
    assert L.canonical_axis((128, 4096, 4095), 1) == (128, 4096, 4095)
    assert L.canonical_axis((4096, 65536), -1) == (4096, 65536, 1)
    assert L.canonical_axis((65536, 4096), 0) == (1, 65536, 4096)
    assert L.canonical_axis((2, 3, 4, 5), 2) == (6, 4, 5)
    with pytest.raises(IndexError):
        L.canonical_axis((2, 3), 2)


def test_product_path_never_imports_the_oracle():
    pkg = os.path.dirname(L.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle.h" not in text, f


def test_short_row_index_division_is_exact():
    """The short-row kernels divide a chunk index e by a row length or a plane
    width d with a multiply and a shift, (e * ceil(2^32 / d)) >> 32; that is
    e // d for every index a chunk holds and every d they are given."""
    import numpy as np
    e = np.arange(0, 8192, dtype=np.uint64)
    for d in range(1, 4097):
        magic = np.uint64(((1 << 32) + d - 1) // d)
        assert np.array_equal((e * magic) >> np.uint64(32), e // np.uint64(d)), d


def test_plane_run_division_is_exact():
    """The plane-run kernel finds plane boundaries in a tile holding k >= 2
    planes of L floats (4 <= L <= 2302: at most half the largest tile of 4608)
    by (e * ceil(2^32 / L)) >> 32 for e up to a tile and a run past it, plus
    64 L where a run start is shifted to stay positive; that is e // L there."""
    import numpy as np
    for d in range(4, (4608 - 3) // 2 + 1):
        e = np.arange(0, 4608 + 72 + 64 * d, dtype=np.uint64)
        magic = np.uint64(((1 << 32) + d - 1) // d)
        assert np.array_equal((e * magic) >> np.uint64(32), e // np.uint64(d)), d


def test_column_group_row_division_is_exact():
    """The column-group scans and reductions find plane boundaries among the
    rows of an item of k >= 2 planes of N rows spanning up to 8 tiles of TR
    rows (S < N <= 4 TR; S = 9, 17 or 33 rows a run for float4, float2 or
    single-float column groups, TR = (128 // G) * S for G groups) by
    (r * ceil(2^32 / N)) >> 32 for r up to 8 tiles and a run past them; that
    is r // N there, for every column count of 3 to 128 the kernels take."""
    import numpy as np
    seen = set()
    for P in range(3, 129):
        V = 4 if P % 4 == 0 else 2 if P % 2 == 0 else 1
        G = P // V
        if G > 32:
            continue
        S = {4: 9, 2: 17, 1: 33}[V]
        rows = (128 // G) * S
        if (rows, S) in seen:
            continue
        seen.add((rows, S))
        r = np.arange(0, 8 * rows + S + 1, dtype=np.uint64)
        for d in range(S + 1, 4 * rows + 1):
            magic = np.uint64(((1 << 32) + d - 1) // d)
            assert np.array_equal((r * magic) >> np.uint64(32), r // np.uint64(d)), (P, d)
