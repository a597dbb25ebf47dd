"""GB300-native paged-KV decode attention.

``paged_kv_cache_265_gb300.pa`` is the Python binding of the C-ABI library
``libpa.so`` (CUDA kernels for sm_103a); ``workload`` holds the seeded input
generator.  Importing this package loads nothing native; ``pa`` loads the
library on first use and raises if it is missing.
"""
