"""Paged KV cache append and paged attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libnk.so`` (hand-written CUDA,
declared in ``include/nk.h``); ``nk`` is its thin ctypes binding and
``workloads`` draws seeded synthetic inputs.  Importing this package does not
load the library; ``nk.load()`` does, and raises if it is missing.
"""

__all__ = ["nk", "workloads"]
