"""GB300-native In-Kernel Broadcast Optimization (IKBO) hot path.

The compute runs in hand-written sm_103a CUDA kernels behind a C ABI
(``include/ikbo.h``, ``libikbo.so``); ``binding`` marshals torch tensors to
it.  Importing this package does not load the library; the first call does,
and raises if the library was not built.  There is no CPU fallback.
"""
__all__ = ["accounting", "inputs"]
