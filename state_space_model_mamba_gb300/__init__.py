"""GB300-native Mamba-2 SSD (state-space duality) chunked selective scan.

The compute lives in ``libssd.so`` (hand-written CUDA for sm_103a behind a
C ABI declared in ``include/ssd.h``); :mod:`state_space_model_mamba_gb300.ssd`
is the thin Python binding that marshals torch tensors into that ABI.
Importing the package loads nothing; the library is opened on first use and
a missing library raises immediately (there is no fallback path).
"""
__all__ = ["ssd", "inputs"]
