"""GB300-native forward pass of one sparsely activated MoE FFN layer.

The compute lives in a C-ABI CUDA library (``csrc/``, declared in
``include/moe.h``); ``token_level_top_gb300.moe`` is the thin ctypes binding
over it.  Importing the package does not load the library: the binding loads
it on first use and raises if it is missing.
"""
__all__ = ["moe", "synth"]
