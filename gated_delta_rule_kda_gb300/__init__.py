"""Kimi Delta Attention (KDA) on one GB300: hand-written sm_103a CUDA kernels
behind a C ABI (``libkda.so``), with a thin ctypes binding.

The binding only marshals arguments; every step of the computation runs in the
library's kernels.  Importing the binding fails loudly when the library has not
been built: there is no CPU fallback.
"""
