"""GB300-native masked multi-head attention over a two-level sparse mask.

The hot path runs in ``libstof.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in include/stof.h).  ``stof`` is its Python binding; the
library is loaded on first use, never at import time.
"""
__all__ = ["stof", "synth"]
