"""B300-native (sm_103a) forward pass of a sparsely-gated Mixture-of-Experts
FFN layer.

The compute runs in libmoe.so (hand-written CUDA, C ABI in include/moe.h);
``binding`` is its ctypes binding, ``layer`` wraps it in a layer object and
``inputs`` draws the seeded synthetic workloads.  Importing the package does
not load the library; the first binding call does, and raises if it is not
built.
"""
__all__ = ["binding", "inputs", "layer"]
