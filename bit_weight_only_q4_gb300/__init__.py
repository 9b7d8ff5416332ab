"""GB300-native 4-bit weight-only linear layers (int4-g128-minmax and NVFP4).

The compute path is a C-ABI shared library of hand-written sm_103a CUDA kernels
(``csrc/``, declared in ``include/q4.h``); :mod:`bit_weight_only_q4_gb300.q4` is the
thin ctypes binding with the same entry-point names.  Importing this package does
not load the library; the first call through the binding does, and raises if the
library has not been built.
"""
__all__ = ["layout", "synth", "q4"]
__version__ = "0.1.0"
