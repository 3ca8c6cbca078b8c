"""Seeded synthetic inputs for the three primitives.

This module draws input values only; it holds none of the arithmetic of the
reductions or the scan, so the oracle and the CUDA path can both be fed from
it.  Every draw is a pure function of (shape, distribution, seed, device type):

* ``uniform01``   torch.rand on a generator seeded with ``seed``.
* ``uniform_pm1`` 2 * torch.rand - 1 (exact in fp32: a power-of-two scale and
  a subtraction of 1 from a value in [0, 2)).
* ``normal``      torch.randn.
* ``harmonic``    x[i] = 1/(i+1), the fp64 reciprocal rounded to fp32 (the
  synthetic fallback input of the "High-Performance Reduction Kernels" README,
  "Layout" section).
* ``const:c``     every element equal to c.
* ``int:lo:hi``   integers drawn uniformly from [lo, hi], stored as fp32.

The generator never reads files and never reaches the network.
"""
from __future__ import annotations

import math

import torch

DISTRIBUTIONS = ("uniform01", "uniform_pm1", "normal", "harmonic", "const", "int")


def _generator(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev.type if dev.type == "cpu" else dev)
    g.manual_seed(int(seed))
    return g


def make(shape, dist: str, seed: int = 0, device="cpu") -> torch.Tensor:
    """Return a contiguous float32 tensor of ``shape`` drawn from ``dist``."""
    shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    n = math.prod(shape)
    dev = torch.device(device)
    if dist == "uniform01":
        return torch.rand(shape, generator=_generator(seed, dev), dtype=torch.float32, device=dev)
    if dist == "uniform_pm1":
        t = torch.rand(shape, generator=_generator(seed, dev), dtype=torch.float32, device=dev)
        return t.mul_(2.0).sub_(1.0)
    if dist == "normal":
        return torch.randn(shape, generator=_generator(seed, dev), dtype=torch.float32, device=dev)
    if dist == "harmonic":
        i = torch.arange(1, n + 1, dtype=torch.float64, device=dev)
        return torch.reciprocal(i).to(torch.float32).reshape(shape)
    if dist.startswith("const:"):
        c = float(dist.split(":", 1)[1])
        return torch.full(shape, c, dtype=torch.float32, device=dev)
    if dist.startswith("int:"):
        _, lo, hi = dist.split(":")
        t = torch.randint(int(lo), int(hi) + 1, shape, generator=_generator(seed, dev),
                          dtype=torch.int32, device=dev)
        return t.to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


# The workloads, by what they are.  ``op`` names the primitive, the other
# keys its arguments; algorithmic_bytes() gives the traffic it must move
# (every input read once, every output written once).
WORKLOADS = {
    "sum_1e6_harmonic": dict(op="sum", shape=(1_000_000,), dist="harmonic", seed=0),
    "sum_1e6_pm1": dict(op="sum", shape=(1_000_000,), dist="uniform_pm1", seed=42),
    "sum_1e9": dict(op="sum", shape=(1_000_000_000,), dist="uniform01", seed=42),
    "axis_128x4096x4095_d1": dict(op="axis", shape=(128, 4096, 4095), dim=1, dist="normal", seed=7),
    "axis_4096x65536_d1": dict(op="axis", shape=(4096, 65536), dim=1, dist="uniform_pm1", seed=11),
    "axis_65536x4096_d0": dict(op="axis", shape=(65536, 4096), dim=0, dist="uniform_pm1", seed=11),
    "rcumsum_32768x32768": dict(op="rcumsum", shape=(32768, 32768), dist="uniform01", seed=3),
    # Few long rows (the look-back scan): one row of 1e9.
    "rcumsum_1x1e9": dict(op="rcumsum", shape=(1, 1_000_000_000), dist="uniform01", seed=3),
    # Other scan forms: forward, exclusive, along a non-last axis.
    "cumsum_fwd_32768x32768": dict(op="cumsum", shape=(32768, 32768), dim=1, reverse=False,
                                   exclusive=False, dist="uniform01", seed=3),
    "cumsum_fwd_excl_1x1e9": dict(op="cumsum", shape=(1, 1_000_000_000), dim=1, reverse=False,
                                  exclusive=True, dist="uniform01", seed=3),
    "cumsum_128x4096x4095_d1": dict(op="cumsum", shape=(128, 4096, 4095), dim=1, reverse=False,
                                    exclusive=False, dist="normal", seed=7),
    # Other reductions on the same shapes.
    "max_1e9": dict(op="reduce", rop="max", shape=(1_000_000_000,), dist="uniform01", seed=42),
    "norm_128x4096x4095_d1": dict(op="reduce", rop="norm", shape=(128, 4096, 4095), dim=1,
                                  dist="normal", seed=7),
    "mean_4096x65536_d1": dict(op="reduce", rop="mean", shape=(4096, 65536), dim=1,
                               dist="uniform_pm1", seed=11),
    "min_65536x4096_d0": dict(op="reduce", rop="min", shape=(65536, 4096), dim=0,
                              dist="uniform_pm1", seed=11),
    # Narrow rows (few columns): the reduction and the scan along dim 1.
    "sum_16x1000000x12_d1": dict(op="reduce", rop="sum", shape=(16, 1_000_000, 12), dim=1,
                                 dist="uniform_pm1", seed=13),
    "cumsum_1024x8192x64_d1": dict(op="cumsum", shape=(1024, 8192, 64), dim=1, reverse=False,
                                   exclusive=False, dist="uniform01", seed=13),
    # The reverse scan of one long row as three passes (reduce-then-scan), for
    # comparison with the single-pass look-back on the same input.
    "rcumsum_1x1e9_rts": dict(op="rcumsum", shape=(1, 1_000_000_000), dist="uniform01", seed=3,
                              strategy=4),
    # Column scans with few column tiles: one pass with warp-split blocks, and
    # too few to fill the GPU (the axis is cut into segments, three passes).
    "cumsum_64x16384x1024_d1": dict(op="cumsum", shape=(64, 16384, 1024), dim=1, reverse=True,
                                    exclusive=False, dist="uniform01", seed=3),
    "cumsum_2x8192x4096_d1": dict(op="cumsum", shape=(2, 8192, 4096), dim=1, reverse=False,
                                  exclusive=True, dist="uniform01", seed=3),
    # Many short rows: the reverse scan of 100-element rows and the sum of
    # 32-element rows (chunks of whole rows staged in shared memory).
    "rcumsum_2000000x100": dict(op="cumsum", shape=(2_000_000, 100), dim=1, reverse=True,
                                exclusive=False, dist="uniform01", seed=3),
    "sum_4000000x32_d1": dict(op="reduce", rop="sum", shape=(4_000_000, 32), dim=1,
                              dist="uniform_pm1", seed=11),
    # Narrow planes (scans and sums along dim 1 with 2-16 columns): many tiny
    # planes, planes one block wide, and one long plane.
    "cumsum_100000x100x3_d1": dict(op="cumsum", shape=(100_000, 100, 3), dim=1, reverse=False,
                                   exclusive=False, dist="uniform01", seed=13),
    "sum_100000x100x3_d1": dict(op="reduce", rop="sum", shape=(100_000, 100, 3), dim=1,
                                dist="uniform_pm1", seed=13),
    "cumsum_4096x4096x2_d1": dict(op="cumsum", shape=(4096, 4096, 2), dim=1, reverse=False,
                                  exclusive=False, dist="uniform01", seed=13),
    "cumsum_1x40000000x4_d1": dict(op="cumsum", shape=(1, 40_000_000, 4), dim=1, reverse=False,
                                   exclusive=False, dist="uniform01", seed=13),
    # Planes of 16 columns (float4 column groups).
    "cumsum_100000x100x16_d1": dict(op="cumsum", shape=(100_000, 100, 16), dim=1, reverse=False,
                                    exclusive=False, dist="uniform01", seed=13),
    # The same calls with caller-provided scratch.
    "rcumsum_1x1e9_ws": dict(op="cumsum", shape=(1, 1_000_000_000), dim=1, reverse=True,
                             exclusive=False, dist="uniform01", seed=3, ws=True),
    "axis_65536x4096_d0_ws": dict(op="reduce", rop="sum", shape=(65536, 4096), dim=0,
                                  dist="uniform_pm1", seed=11, ws=True),
}

# The 1D sweep sizes of the sum benchmark (uniform[0,1), seed 42).
SUM_SWEEP = (10_000, 100_000, 1_000_000, 10_000_000, 100_000_000, 500_000_000, 1_000_000_000)


def canonical_axis(shape, dim):
    """(outer, reduce, inner) of a contiguous tensor reduced along ``dim``."""
    shape = tuple(int(s) for s in shape)
    dim = dim % len(shape)
    outer = math.prod(shape[:dim])
    inner = math.prod(shape[dim + 1:])
    return outer, shape[dim], inner


def algorithmic_bytes(w: dict) -> int:
    """Bytes the primitive must move: read each input once, write each output once."""
    n = math.prod(w["shape"])
    if w["op"] == "sum":
        return 4 * n + 4
    if w["op"] in ("axis", "reduce") and "dim" in w:
        outer, _, inner = canonical_axis(w["shape"], w["dim"])
        return 4 * n + 4 * outer * inner
    if w["op"] == "reduce":
        return 4 * n + 4
    if w["op"] in ("rcumsum", "cumsum"):
        return 8 * n
    raise ValueError(w["op"])
