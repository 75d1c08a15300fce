"""GB300-native compressed sparse attention (c4a / c128a) for decode and
chunked prefill: a C-ABI CUDA library (``libv4a``) and a thin ctypes binding.

Importing the package does not load the CUDA library; ``v4a`` (the binding)
loads it on first use and raises if it is missing.
"""
