"""MoBA (Mixture of Block Attention) forward pass for GB300 (sm_103a).

The compute lives in ``libmoba_gb300.so`` (hand-written CUDA behind a C ABI,
declared in ``include/moba.h``); this package is the thin Python binding.
"""
