"""GB300-native XAttention block-sparse attention for chunked prefill.

The compute path is the CUDA library ``libxattn`` (C ABI, see
``include/xattn.h``); ``xattention_block_sparse_gb300.xattn`` binds it with
ctypes.  Importing this package loads nothing: the library is opened on first
use and a missing library raises instead of falling back to anything else.
"""
