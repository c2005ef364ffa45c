"""GB300-native paged KV cache decode path.

The compute lives in ``libpagedkv.so`` (CUDA for sm_103a behind a C ABI,
declared in ``include/pagedkv.h``); ``paged_kv_cache_33_gb300.pagedkv`` is the
thin ctypes binding with the same names.  ``workloads`` draws the seeded
synthetic inputs.  Importing the package loads nothing; the binding loads the
library on first use and raises if it is missing.
"""

__all__ = ["pagedkv", "workloads"]
