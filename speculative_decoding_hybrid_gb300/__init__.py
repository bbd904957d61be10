"""gdnspec: K-draft MTP speculative verification over GatedDeltaNet layers on
one GB300 (sm_103a).

The compute lives in ``libgdnspec.so`` (CUDA kernels + host planner behind the
C ABI of ``include/gdnspec.h``).  ``binding`` is the thin ctypes layer with
the same function names; ``step`` groups the per-transaction call sequence.
Both fail at import when the library has not been built.
"""
__all__ = ["binding", "step", "build"]
