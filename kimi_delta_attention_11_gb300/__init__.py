"""GB300 (sm_103a) Kimi Delta Attention forward: Python binding of libkda_gb300.so.

The compute path is the CUDA library declared in include/kda.h; this package only
marshals tensors into its C ABI.  Build the library with ``build.build_library()``
(or ``__graft_entry__.build()``) before use.
"""
from ._native import (DTYPE_CODES, KdaError, KdaLibraryMissing, build_chunk_index, decode, fwd,
                      get_device_status, launch_count, library_path, load_library, schedule,
                      selftest_umma, status_string, workspace_bytes)

__all__ = ["fwd", "decode", "workspace_bytes", "launch_count", "schedule", "build_chunk_index",
           "get_device_status", "status_string", "load_library", "library_path", "selftest_umma",
           "KdaError", "KdaLibraryMissing", "DTYPE_CODES"]
