"""Multi-scale deformable attention (MSDA) for GB300 (sm_103a).

The compute path is ``libmsda.so``: hand-written CUDA kernels behind a C ABI
(declared in ``include/msda.h``). ``binding`` is a thin ctypes layer over it
that passes device pointers and the current CUDA stream; ``workloads`` draws
seeded synthetic operands. Importing this package loads nothing: the library is
opened on the first call and a missing library is an error, never a fallback.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads"]
