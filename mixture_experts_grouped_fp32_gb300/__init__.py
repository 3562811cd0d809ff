"""GB300-native (sm_103a) forward pass of a Mixture-of-Experts FFN layer.

The compute path is the C-ABI library ``libmoe.so`` (hand-written CUDA for sm_103a, declared in
``include/moe.h``); ``moe`` is its thin ctypes binding and ``workloads`` draws seeded synthetic
inputs.  Importing this package does not load the library: the binding loads it on first use and
raises if it has not been built.
"""
__all__ = ["moe", "workloads"]
