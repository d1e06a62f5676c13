"""B300-native curvature-whitened truncated SVD with global rank allocation.

The compute path is libkfsvd.so (hand-written CUDA for sm_103a, C ABI in include/kfsvd.h);
``kfsvd`` binds it with ctypes and ``pipeline`` strings its five steps over a workload.
"""
from . import kfsvd  # noqa: F401
