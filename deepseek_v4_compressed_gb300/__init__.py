"""GB300-native decode path of DeepSeek-V4 compressed sparse attention.

The compute runs in the CUDA library ``libdsv4.so`` (sm_103a kernels behind a
C ABI declared in ``include/dsv4.h``); ``binding`` is its thin ctypes binding.
"""
