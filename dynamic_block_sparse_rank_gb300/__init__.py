"""Dynamic block-sparse attention for video DiTs on GB300 (sm_103a).

The compute lives in libsda.so (C ABI, include/sda.h); `sda` is its thin
ctypes binding and `inputs` draws the seeded synthetic workloads.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "sda", "build"]
