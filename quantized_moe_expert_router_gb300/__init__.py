"""GB300-native routed NVFP4 MoE FFN (router, top-k, SwiGLU experts, combine).

The compute path lives in ``csrc/`` (CUDA for sm_103a behind a C ABI declared
in ``include/moe.h``); ``moe`` is the thin ctypes binding with the same names.
``synth`` generates seeded synthetic inputs.
"""
