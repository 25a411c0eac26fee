"""GB300-native (sm_103a) jagged index + embedding hot path of FreeScale-style training.

Modules:
  binding   -- ctypes binding of the C ABI (include/fs_jagged.h) over torch tensors
  pipeline  -- one training iteration sequenced over preallocated device buffers
  synthetic -- seeded synthetic inputs shaped like the FreeScale workloads
  build     -- in-tree nvcc build of libfsjagged.so
"""
__all__ = ["binding", "pipeline", "synthetic", "build"]
