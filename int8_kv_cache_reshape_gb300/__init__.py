"""GB300-native quantized paged-KV attention (sm_103a).

The compute lives in the C-ABI library ``libkvq.so`` built from ``csrc/``
(see ``include/kvq.h``); ``kvq`` is its thin ctypes binding.  Importing this
package loads nothing: ``from int8_kv_cache_reshape_gb300 import kvq`` does,
and fails loudly when the library has not been built.
"""
__all__ = ["kvq", "workloads", "build"]
