"""GB300 sampling hot path of speculative decoding (Markov-head draft +
lossless verify) behind a C ABI (include/spec.h).

Submodules:
  build      -- in-tree nvcc build of libspec.so (sm_103a)
  _lib       -- ctypes binding, same names as the C entry points
  engine     -- torch-side buffers and one-cycle helper
  workloads  -- seeded synthetic inputs (no method arithmetic)

Importing the package does not load the CUDA library; the first call through
``_lib`` does, and raises if it is missing.
"""
