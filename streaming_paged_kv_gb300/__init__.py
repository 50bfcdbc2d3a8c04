"""GB300-native two-stream paged KV cache with per-frame paged attention.

The compute path is the C-ABI library ``libkvc.so`` (CUDA kernels for sm_103a
plus a C++ page allocator); ``streaming_paged_kv_gb300.kvc`` binds it with
ctypes.  Importing this package does not load the library; importing ``kvc``
does, and fails loudly if it has not been built.
"""
