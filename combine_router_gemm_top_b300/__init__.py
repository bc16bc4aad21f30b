"""B300-native (sm_103a) mixture-of-experts layer forward pass.

The hot path -- route, dispatch layout, permute, grouped SwiGLU FFN,
combine -- runs in hand-written CUDA kernels behind the C-ABI library
``libmoe.so`` (declared in include/moe.h).  This package holds the library's
sources, a thin ctypes binding with the same entry-point names, a host-side
layer object that owns device buffers, and the seeded synthetic workloads.
"""
__all__ = ["workloads"]
