"""B300-native top-2 sparse MoE feed-forward layer (Mixtral shape).

The compute lives in ``libmoe.so`` (hand-written CUDA for sm_103a, C ABI in
``include/moe.h``); ``sparse_mixture_experts_53_b300.moe`` is its ctypes
binding and ``sparse_mixture_experts_53_b300.build`` compiles it. Neither is
imported here, so that the build can run before the library exists.
"""
