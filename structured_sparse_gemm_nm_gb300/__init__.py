"""N:M structured-sparsity hot path for NVIDIA GB300 (sm_103a).

The computation lives in the CUDA library ``lib/libnm.so`` (C ABI:
``include/nm.h``); :mod:`.binding` exposes its entry points to Python with
the same names, and :mod:`.inputs` draws the seeded synthetic workloads.
Importing the package does not load the library; the first call does, and
fails loudly if it was not built.
"""
from . import inputs  # noqa: F401

__all__ = ["binding", "inputs"]
