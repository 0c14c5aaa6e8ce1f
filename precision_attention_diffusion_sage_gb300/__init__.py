"""Quantized (Sage-style) attention forward for GB300 (sm_103a).

The compute path is the C-ABI library ``libsage.so`` (hand-written CUDA
kernels); ``binding`` is a thin ctypes layer over it with the same names.
Importing this package does not load the library; ``binding`` does, and it
raises if the library is missing.
"""
__all__ = ["binding", "inputs"]
