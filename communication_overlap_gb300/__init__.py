"""FlashOverlap's signaled GEMM + reorder hot path, GB300-native (sm_103a).

The compute path lives in ``libfo.so`` (CUDA kernels behind a C ABI, see
``include/fo.h``); ``communication_overlap_gb300.fo`` is the thin ctypes
binding with the same function names.  Importing this package loads
nothing; the binding loads the library on first use and raises if it is
missing.
"""
