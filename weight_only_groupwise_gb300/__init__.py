"""Groupwise int4/int5 small-batch projection for GB300 (sm_103a).

The compute lives in libnq.so (hand-written CUDA, C ABI in include/nq.h); ``nq`` is its thin
ctypes binding. Build the library with ``weight_only_groupwise_gb300.build.build()``.
"""
from . import nq  # noqa: F401
