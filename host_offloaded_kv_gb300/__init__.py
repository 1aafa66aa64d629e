"""CLO decode-step hot path for GB300 (sm_103a).

CPU-light KV-cache offloading: full K/V in pinned host memory, hash-code top-k
selection (10 %), head-wise reuse of the previous on-GPU selection, persistent
heads resident in HBM, zero-copy GPU fetch of missed rows and split-K sparse
attention -- all in the CUDA library behind the C ABI of ``include/clo.h``.
``clo`` is the Python binding (ctypes, marshalling only); ``synth`` generates the
seeded synthetic workloads.
"""
from . import clo  # noqa: F401  (the binding loads libclo.so lazily and raises if it is missing)
from .clo import CLOContext, CLOError  # noqa: F401

__all__ = ["clo", "CLOContext", "CLOError"]
