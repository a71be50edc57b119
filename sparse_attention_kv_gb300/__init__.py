"""GB300-native query-sparse-attention block selection.

The compute path lives in ``libqsa.so`` (CUDA, sm_103a) behind the C ABI of
``include/qsa.h``; ``sparse_attention_kv_gb300.qsa`` is its thin ctypes
binding.  Importing this package does not load the library; the first call
into the binding does, and fails loudly if the library was not built.
"""
__all__ = ["inputs", "qsa"]
