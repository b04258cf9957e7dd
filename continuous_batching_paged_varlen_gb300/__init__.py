"""Paged, mixed-batch (continuous-batching) attention for one GB300.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/mb.h``); ``binding`` is a thin
ctypes layer with the same call names. ``workloads`` draws seeded synthetic
inputs and ``counters`` holds the bench's algorithmic byte / FLOP counts.

Importing this package does not load the library; ``binding.lib()`` does,
and raises if the compiled library is missing (there is no fallback path).
"""

__all__ = ["binding", "workloads", "counters"]
