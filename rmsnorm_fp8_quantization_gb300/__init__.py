"""Fused LayerNorm / RMSNorm forward (+FP8 E4M3 delayed or MXFP8 output) and
backward (+fused residual-gradient add) for GB300 (sm_103a).

The compute path is the C-ABI library ``libgbnorm.so`` built from ``csrc/``;
``gbnorm`` is its ctypes binding.
"""
