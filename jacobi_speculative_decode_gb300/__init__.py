"""GB300-native XPress Jacobi refinement pass.

The compute path is the CUDA library ``libxp.so`` (hand-written sm_103a
kernels behind a C ABI declared in ``include/xp.h``); ``xp`` is its thin
ctypes binding and ``inputs`` the seeded synthetic-input generator.
"""
