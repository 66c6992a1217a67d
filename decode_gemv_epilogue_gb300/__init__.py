"""Decode-path GEMV with a fused element-wise epilogue and a signed Walsh-Hadamard
prologue, written for GB300 (sm_103a).

The compute lives in the C-ABI library ``libgemvfuse.so`` (CUDA kernels in ``csrc/``,
declared in ``include/gemvfuse.h``).  ``gemvfuse`` is the thin ctypes binding over it;
``synth`` draws the seeded synthetic inputs.  Importing this package does not load the
library; importing ``gemvfuse`` does, and fails loudly when it has not been built.
"""
