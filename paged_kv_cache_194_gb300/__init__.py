"""GB300-native paged KV cache decode attention.

The compute path is the C-ABI library ``libpkv.so`` (hand-written CUDA for
sm_103a, sources under ``csrc/``); this package holds its thin Python binding,
the host-side block manager and the seeded workload generators.  The library
is loaded on first use and a missing build raises immediately -- there is no
CPU fallback.
"""
