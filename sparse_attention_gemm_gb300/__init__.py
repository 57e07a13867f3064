"""GB300-native (sm_103a) DSA forward hot path behind a C ABI.

The compute lives in ``libdsa.so`` (hand-written CUDA kernels, built from
``csrc/`` by ``build.py``); ``ops`` is a thin ctypes binding with the same
entry-point names.  Importing this package does not load the library; the
first call into ``ops`` does, and raises if it is missing.
"""
__all__ = ["workloads"]
