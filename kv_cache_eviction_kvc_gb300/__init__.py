"""Budgeted-KV decode step and LaProx prefill scorer on GB300 (sm_103a).

The compute lives in libkvc (``csrc/``, C ABI in ``include/kvc.h``); ``kvc``
is its thin ctypes binding, ``state`` allocates device memory for a decode
stream, ``workloads`` draws the seeded synthetic inputs and ``dist`` holds
the multi-process plumbing (the layer-sharded prefill exchange).
"""
__all__ = ["kvc", "state", "workloads", "dist"]
