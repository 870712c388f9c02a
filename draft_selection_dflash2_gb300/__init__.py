"""DFlash 2 draft-block head for NVIDIA GB300 (sm_103a).

The compute path lives in libdflash2.so (hand-written CUDA behind a C ABI, see
include/dflash2.h); ``api`` is its thin Python binding and ``synth`` the seeded
synthetic-input generator.  Importing the package loads nothing: the library
is loaded (and must exist) on first use of ``api``.
"""
__all__ = ["api", "synth"]
