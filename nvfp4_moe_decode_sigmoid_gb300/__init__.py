"""GB300-native small-batch decode of a Flint-style NVFP4 MoE layer.

The compute lives in ``libflint.so`` (hand-written CUDA for sm_103a behind a
C ABI declared in ``include/flint.h``); ``flint`` is its thin Python binding.
"""
