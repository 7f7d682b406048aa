"""GB300-native routed NVFP4 SiTU MoE forward.

The compute lives in a C-ABI CUDA library (``csrc/`` -> ``lib/libnvfp4moe.so``,
declared in ``include/nvfp4moe.h``); :mod:`nvfp4_routed_moe_gb300.api` is a
thin ctypes binding with the same entry-point names.  Importing this package
does not load the library; the first call through the binding does, and it
raises if the library is missing (there is no CPU fallback).
"""
__all__ = ["api", "inputs", "build"]
