"""NVFP4 decode-projection library for one GB300 (sm_103a).

The compute lives in the C-ABI shared library ``libaq.so`` (declared in
``include/aq.h``); ``nvfp4_block_scaled_aq_gb300.aq`` is its thin ctypes
binding.  Importing this package loads nothing: the library is opened on
first use of the binding, which raises if the CUDA build is missing.
"""
