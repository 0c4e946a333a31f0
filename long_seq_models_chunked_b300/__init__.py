"""B300-native (sm_103a) chunked test-time-training fast-weight layer.

The layer lives in a C-ABI CUDA library (include/ttt.h); ``abi`` is its thin
ctypes binding, ``synth`` the seeded synthetic workloads and ``accounting`` the
fixed FLOP/byte counts used for throughput and roofline figures.
"""
__all__ = ["abi", "synth", "accounting"]
