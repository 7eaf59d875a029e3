"""GB300-native paged KV cache: the KV-cache write and PagedAttention.

The compute path lives in ``csrc/`` (CUDA for sm_103a) behind the C ABI of
``include/pkv.h``; ``pkv`` is a thin ctypes binding with the same names.
Importing this package loads nothing: ``pkv`` loads ``libpkv.so`` on first use
and raises if it is missing.
"""
__all__ = ["workloads", "pkv"]
