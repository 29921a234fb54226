"""GB300-native DTensor tensor-parallel linear and layout transforms.

The compute lives in ``libdt.so`` (CUDA kernels for sm_103a behind a C ABI
declared in ``include/dt.h``); this package is a thin ctypes binding over it.
The library is loaded on first use and a missing build raises immediately:
there is no CPU fallback.
"""
