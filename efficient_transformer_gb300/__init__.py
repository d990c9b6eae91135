"""GB300-native fused linear attention (forward and backward) and the low-rank projection.

The compute path is a C-ABI shared library built from hand-written sm_103a CUDA
(``csrc/``); ``efficient_transformer_gb300.la`` is its thin Python binding.  Importing
this package loads nothing: the library is opened on the first call and a missing
library raises an error (there is no fallback).
"""
__all__ = ["la", "inputs"]
