"""libreduce for GB300 (sm_103a): fp32 sum, axis sum and reverse cumulative sum.

The compute runs in hand-written CUDA kernels behind a C ABI
(``include/libreduce.h``); this package holds those sources (``csrc/``), the
in-tree build step and a thin ctypes binding.  ``inputs`` holds the seeded
synthetic input generator.
"""
