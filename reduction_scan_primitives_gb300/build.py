"""In-tree build of libreduce.so (nvcc, sm_103a only).

Compiles each translation unit under csrc/ in parallel and links lib/libreduce.so
inside this package.  The CUDA runtime is linked statically, so the
library needs only the NVIDIA driver at run time.  ptxas resource usage
(registers, spills, shared memory) of every kernel is written to
_build/ptxas.log.

build(debug=True) makes lib/libreduce_debug.so instead: the same entry points
with device-side checks of every kernel access against the call's buffers
(LR_DEBUG; relocatable device code, so all kernels share one record of the
registered ranges).  It is for finding a bad index, not for timing.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "lib", "libreduce.so")
DEBUG_LIB = os.path.join(HERE, "lib", "libreduce_debug.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
SOURCES = ["lr_api.cu", "lr_reduce.cu", "lr_scan.cu", "lr_scan_cols_lb.cu", "lr_rows_short.cu", "lr_narrow.cu",
           "lr_planes_scan.cu", "lr_planes_reduce.cu", "lr_planes_lb.cu",
           "lr_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-Wall,-fvisibility=hidden",
              "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libreduce")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "libreduce.h"))
    files.append(__file__)
    return files


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build libreduce.so (debug: libreduce_debug.so) if it is missing or older
    than its sources; returns its path."""
    lib, bdir = (DEBUG_LIB, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    nvcc = _nvcc()
    flags = [*NVCC_FLAGS, "-DLR_DEBUG=1", "-rdc=true"] if debug else NVCC_FLAGS

    def compile_one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    with open(os.path.join(bdir, "ptxas.log"), "w") as f:
        for (_, log), src in zip(results, SOURCES):
            f.write(f"==== {src}\n{log}\n")
    tmp = lib + f".tmp{os.getpid()}"
    link = [nvcc, "-shared", *ARCH, *(["-rdc=true"] if debug else []), "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(open(os.path.join(bdir, "ptxas.log")).read())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
