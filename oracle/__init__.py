"""CPU oracle for block-diagonal causal attention over packed sequences.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` import this package.  It shares no code with the CUDA
path and imports nothing from it.
"""
from .blockdiag import (  # noqa: F401
    PAD_DOC_ID,
    blockdiag_sdpa_backward,
    blockdiag_sdpa_forward,
    doc_ids_from_cu_seqlens,
    segment_cu_seqlens,
)
