"""GB300-native (sm_103a) W8A8 quantized verify pass for speculative decoding.

The computation lives in ``libqv.so`` (CUDA kernels behind the C ABI of
``include/qv.h``); ``qv`` is its thin ctypes binding, ``synth`` draws the
seeded synthetic workloads, ``build`` compiles the library with nvcc.
Submodules are imported on demand: ``from quantized_verification_gb300 import qv``.
"""
__all__ = ["qv", "synth", "build"]
