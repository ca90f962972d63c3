"""GB300-native fused contraction + activation/normalisation operators.

The compute lives in ``libgf.so`` (hand-written CUDA for sm_103a behind a C
ABI declared in ``include/gf.h``); :mod:`.binding` marshals torch tensors into
that ABI.  Importing this package does not load the library; the first call
does, and raises if it is missing.
"""
__all__ = ["binding", "synth"]
