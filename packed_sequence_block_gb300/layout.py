"""Row-layout helpers on the device: document ids from lengths, document
positions and validity, the position check, and the key/value rows the local
queries of an interval need.

Thin wrappers over the C ABI (``include/bd_attn.h``): they allocate the
outputs and marshal arguments; every step runs in the library's kernels.
Pages: "nemo_automodel.components.models.glm5_next.cp" (doc_ids_from_seq_lens),
"nemo_automodel.components.models.inkling2.context_parallel"
(unpack_row_layout, validate_document_positions) and
"nemo_automodel.components.distributed.blockdiag_cp" (the needed-only K/V
exchange of cp_blockdiag_sdpa).
"""
from __future__ import annotations

import torch

from . import _native as N
from .attention import check_device_status, device_status_word


def doc_ids_from_seq_lens(seq_lens, seq_len: int, padding_value: int = -1000,
                          device=None) -> torch.Tensor:
    """Document ids [B, seq_len] (int32, 0 == padding) from lengths [B, documents].

    Entries equal to ``padding_value`` are not documents.  Raises ValueError
    for a negative length or a row longer than ``seq_len`` (this reads the
    device status word back, so it synchronises).
    """
    dev = device if device is not None else (
        seq_lens.device if isinstance(seq_lens, torch.Tensor) and seq_lens.is_cuda else "cuda")
    lens = torch.as_tensor(seq_lens).to(device=dev, dtype=torch.int32)
    if lens.dim() == 1:
        lens = lens.unsqueeze(0)
    if lens.dim() != 2:
        raise ValueError("seq_lens must be [documents] or [batch, documents]")
    lens = lens.contiguous()
    B, ndocs = lens.shape
    ids = torch.empty((B, seq_len), dtype=torch.int32, device=lens.device)
    N.bd_doc_ids_from_seq_lens(lens, B, ndocs, seq_len, padding_value, ids,
                               device_status_word(lens.device))
    check_device_status(lens.device)
    return ids


def position_ids_from_doc_ids(doc_ids: torch.Tensor):
    """(positions int32 [B, S], keep bool [B, S]) for document ids [B, S] or [S]."""
    ids = doc_ids.reshape(-1, doc_ids.shape[-1]).to(torch.int32).contiguous()
    B, S = ids.shape
    pos = torch.empty((B, S), dtype=torch.int32, device=ids.device)
    keep = torch.empty((B, S), dtype=torch.bool, device=ids.device)
    N.bd_position_ids_from_doc_ids(ids, B, S, pos, keep)
    return pos, keep


def document_position_violations(keep: torch.Tensor, positions: torch.Tensor) -> torch.Tensor:
    """First offending column of each row (int32 [B], -1 where the row is valid)."""
    k = keep.reshape(-1, keep.shape[-1]).to(torch.bool).contiguous()
    p = positions.reshape(-1, positions.shape[-1]).to(torch.int32).contiguous()
    if k.shape != p.shape:
        raise ValueError("keep and positions must have the same shape")
    B, S = k.shape
    bad = torch.empty((B,), dtype=torch.int32, device=k.device)
    N.bd_validate_document_positions(k, p, B, S, bad, None)
    return bad


def validate_document_positions(keep: torch.Tensor, positions: torch.Tensor) -> None:
    """Raise ValueError unless positions step by one inside documents and reset to 0
    at a new document (the first valid span of a row may start at any offset >= 0;
    a gap cannot resume an old document).  Synchronises."""
    bad = document_position_violations(keep, positions).cpu()
    rows = torch.nonzero(bad >= 0).reshape(-1)
    if rows.numel():
        r = int(rows[0])
        raise ValueError(f"document positions are not valid: row {r}, column {int(bad[r])}")


def kv_needed_range(seg, seg_ids, nseg, L: int, seq_start: int, shards: bool = True):
    """(range int32 [B, 2], shard_rows int32 [B, ceil(S/L)] or None) for the local
    queries [seq_start, seq_start + L) of rows segmented by segment_cu_seqlens."""
    B, S = seg_ids.shape
    rng = torch.empty((B, 2), dtype=torch.int32, device=seg.device)
    rows = (torch.empty((B, -(-S // L)), dtype=torch.int32, device=seg.device)
            if shards else None)
    N.bd_kv_needed_range(seg, seg_ids, nseg, B, S, L, seq_start, rng, rows)
    return rng, rows
