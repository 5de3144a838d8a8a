"""GB300-native (sm_103a) Gemma-4 E-series dual-geometry attention path.

The compute lives in ``libg4attn.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/g4attn.h``).  ``g4attn`` is the thin ctypes binding;
``workloads`` holds the seeded synthetic inputs.  Importing this package does
not load the library; ``g4attn.lib()`` does, and raises if it is missing.
"""
