"""GB300-native paged KV-cache attention.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``include/pkv.h``); :mod:`paged_kv_cache_pg_gb300.pkv` is its thin
ctypes binding.  Importing this package loads nothing; import ``pkv`` to load
the library.
"""
