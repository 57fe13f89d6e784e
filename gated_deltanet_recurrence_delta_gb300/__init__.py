"""Gated DeltaNet layer hot path for GB300 (sm_103a).

``gdn``     -- thin ctypes binding of the C-ABI library ``libgdn.so`` (CUDA kernels)
``inputs``  -- seeded synthetic inputs shared by tests and benchmarks
``build``   -- nvcc build of ``libgdn.so`` (in-tree)
"""
