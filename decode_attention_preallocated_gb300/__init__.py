"""Length-aware GQA decode attention over a preallocated KV cache (GB300).

The computation lives in libfd.so (hand-written CUDA for sm_103a, C ABI in
include/fd.h); ``fd`` is its ctypes binding and ``build`` compiles it.
``workloads`` makes seeded synthetic inputs.  Importing the package does not
load the library; the first call does, and raises if it is not built.
"""
from .fd import (FD_KERNEL_AUTO, FD_KERNEL_SIMT, FD_KERNEL_TC, FdError,  # noqa: F401
                 Workspace, decode, decode_gather, decode_int8, plan)

__all__ = ["decode", "decode_int8", "decode_gather", "Workspace", "plan",
           "FdError", "FD_KERNEL_AUTO", "FD_KERNEL_SIMT", "FD_KERNEL_TC"]
