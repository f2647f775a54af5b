"""Block-diagonal (per-document) causal attention over packed sequences, for GB300.

The compute path is a C-ABI CUDA library (``libbd_attn.so``, built for
sm_103a from ``csrc/``); this package loads it with ctypes and passes it
torch-owned device buffers.  There is no CPU fallback: every entry point
raises if the library is missing.
"""
