"""B300-native forward pass of a token-choice top-k MoE SwiGLU layer.

The compute runs in hand-written sm_103a CUDA kernels behind a C ABI
(``include/moe.h``, built as ``libmoe_b300.so`` in this package); ``api``
is the thin Python binding over it.
"""
