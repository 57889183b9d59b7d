"""GB300 (sm_103a) online KV-cache compression and compressed-cache decode attention.

``tq`` is the ctypes binding of the C ABI (``include/tq.h``); ``workloads``
generates the seeded synthetic inputs; ``build`` compiles ``libtq.so``.
"""
