"""Gated DeltaNet (GDN) token-mixing core for NVIDIA B300 (sm_103a).

The compute lives in ``libgdn.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/gdn.h``); ``gdn`` is the thin ctypes binding over it.
Importing the package does not load the library: the first call does, and it
raises if the library is missing.
"""
from .inputs import WORKLOADS  # noqa: F401
