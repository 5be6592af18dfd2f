"""GB300-native (sm_103a) fused multi-head attention backward pass.

The compute path is a C-ABI shared library of hand-written CUDA kernels
(``csrc/``); ``binding`` marshals arguments to it through ctypes.  Importing
this package does not load the library; ``binding.load()`` does, and raises if
the library is missing.
"""
__all__ = ["binding", "build", "workloads", "flops"]
