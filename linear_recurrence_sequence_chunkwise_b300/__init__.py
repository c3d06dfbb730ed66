"""RetNet multi-scale retention core on one B300 (sm_103a).

The compute lives in a C-ABI shared library of hand-written CUDA kernels
(``csrc/``, header ``include/retention.h`` at the repository root).  The
Python side is a thin ctypes binding (:mod:`.binding`) that only marshals
pointers, sizes and streams; PyTorch supplies device memory and streams.
Importing this package loads nothing; the binding loads the library on first
use and raises if it is missing.
"""
__all__ = ["binding", "inputs"]
