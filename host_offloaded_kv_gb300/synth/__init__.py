"""Seeded synthetic inputs for the CLO decode workloads.

The generator is a small C library (``synth.c``) loaded with ctypes.  It holds
none of the method's arithmetic: it produces keys, values, queries and the hash
projection, and both the CUDA library and the CPU oracle take their inputs from
it.  See ``workloads.py`` for the five named workloads.
"""
from .synth import (  # noqa: F401
    Synth,
    load_synth,
    bf16_to_float,
    float_to_bf16,
)
from .workloads import WORKLOADS, Workload, get_workload  # noqa: F401
