"""tovl: producer-row movement fused with a tcgen05 bf16 GEMM on one GB300.

The library itself is ``libtovl.so`` (C ABI in ``include/tovl.h``), built by
``consumer_movement_gemm_gb300.build``; ``consumer_movement_gemm_gb300.tovl``
is its ctypes binding.  Importing this package does not load the library.
"""
from .tovl import Handle, TovlError, dispatch_rows, load  # noqa: F401

__all__ = ["Handle", "TovlError", "dispatch_rows", "load"]
