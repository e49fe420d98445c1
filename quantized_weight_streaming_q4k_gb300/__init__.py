"""Quantized weight streaming for single-token decode on GB300 (sm_103a).

Modules:
  ops    -- torch-facing binding of the C ABI in include/qws.h (libqws.so)
  synth  -- seeded synthetic inputs (numpy), shared by tests and the benchmark
  build  -- in-tree nvcc build of libqws.so
"""
__version__ = "0.1.0"
