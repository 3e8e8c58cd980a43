"""GB300-native (sm_103a) TetraJet-v2 NVFP4 linear layer.

The compute path is the CUDA library ``libtj.so`` built from ``csrc/`` and
reached through its C ABI; ``nvfp4_bit_fully_gb300.tj`` is the thin ctypes
binding (argument marshalling only).  ``workloads`` draws the seeded
synthetic inputs.  Importing this package does not load the library; the
binding raises if the library is missing, and there is no CPU fallback.
"""
__all__ = ["tj", "workloads"]
