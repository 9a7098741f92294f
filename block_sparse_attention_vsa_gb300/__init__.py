"""GB300-native (sm_103a) block-sparse attention forward: VSA look-up tables and Jenga
block bitmaps.

The computation runs in hand-written CUDA kernels behind a C ABI
(``include/vsa.h``, built into ``libvsa_gb300.so``); :mod:`.binding` is the thin
Python layer over that library.  Importing this package does not load the
library; the first call into :mod:`.binding` does, and fails loudly if it has
not been built.
"""
__all__ = ["binding", "workloads"]
