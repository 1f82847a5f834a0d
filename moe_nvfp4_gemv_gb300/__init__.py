"""libfp4gemv: NVFP4 (W4A16) small-M GEMV kernels for GB300 (sm_103a).

The compute lives in the C-ABI shared library ``libfp4gemv.so`` built from
``moe_nvfp4_gemv_gb300/csrc``; ``moe_nvfp4_gemv_gb300.fp4gemv`` is the thin
ctypes binding with the same call names.  Importing this package does not
load the library (so the seeded input generators in ``synth`` work on a
machine without a GPU); importing ``fp4gemv`` does, and fails loudly when the
library is missing.
"""
__all__ = ["synth"]
