"""Gated DeltaNet (GDN) layer core forward on GB300 (sm_103a).

``build.build()`` compiles ``libgdn.so`` in-tree; ``gdn`` is its ctypes
binding (the C ABI of ``include/gdn.h``); ``workloads`` holds the seeded
synthetic inputs.
"""
