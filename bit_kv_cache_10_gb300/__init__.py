"""TurboQuant packed KV cache for GB300 (sm_103a).

The CUDA library ``libtq.so`` (C ABI in ``include/tq.h``) holds every step of
the hot path; ``native`` is its ctypes binding and ``cache`` a thin torch
wrapper that owns the device buffers.  ``synth`` draws the seeded synthetic
workloads.  Build the library with ``bit_kv_cache_10_gb300.build.build()``.
"""
from . import native  # noqa: F401
