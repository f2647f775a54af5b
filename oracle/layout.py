"""Oracle for the packed-row layout helpers: plain CPU statements, pure Python loops.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import or run this module.  The product path (the
CUDA library and its Python binding) never imports it, and this module
imports nothing from the product package.

What it follows (NeMo Automodel API reference pages):

* "nemo_automodel.components.models.glm5_next.cp", ``doc_ids_from_seq_lens``:
  per-document lengths [batch, documents], padded with ``padding_value``
  (default -1000), become document ids [batch, sequence].
* "nemo_automodel.components.models.inkling2.context_parallel",
  ``unpack_row_layout`` (boolean validity and integer document positions
  [batch, sequence], padding decided from the lengths, never from token ids)
  and ``validate_document_positions(keep, positions)``: inside a document the
  position grows by one per token, a new document starts at zero, a shard may
  begin partway through a document (its first real span may start at a
  non-zero offset, also after left padding), and a gap cannot resume an old
  document.
* "nemo_automodel.components.distributed.blockdiag_cp", ``cp_blockdiag_sdpa``:
  keys and values reach the local queries by all-gather "or a needed-only
  halo/a2a exchange"; the keys a local query needs are the keys its
  per-document causal mask allows.

Readings where the pages are silent (each is listed in the design notes):

* ``doc_ids_from_seq_lens``: entries equal to ``padding_value`` are not
  documents and take no number, wherever they stand; the other entries are
  documents numbered 1..n in order (a zero-length document still takes its
  number); any other negative length, or a total past ``seq_len``, is an
  error; positions past the last document are padding (id 0);
* document positions come from the document ids: a document is a maximal
  run of equal non-zero ids, its tokens get 0, 1, 2, ...; padding tokens
  (id 0) get position 0 and validity false;
* ``validate_document_positions``: among the valid tokens of a row, in order,
  the first may carry any position >= 0; each later one must carry 0, or its
  predecessor's position + 1 when it directly follows that predecessor;
  after a gap (invalid tokens between the two) it must carry 0.  The result
  here is the first offending column of each row, or -1;
* the needed key/value rows of the local queries [seq_start, seq_start + L)
  are the union of their masks: [lo, hi) with lo the start of the segment of
  the first non-padding local query and hi one past the last non-padding
  local query; empty (lo = hi = seq_start) when every local query is padding.
  With the row cut into consecutive shards of L positions, the rows needed
  from shard r are the part of [lo, hi) inside that shard.
"""
from __future__ import annotations

import numpy as np

from .blockdiag import PAD_DOC_ID, doc_ids_from_cu_seqlens


def doc_ids_from_seq_lens(seq_lens, seq_len: int, padding_value: int = -1000) -> np.ndarray:
    """Document ids [B, seq_len] from per-document lengths [B, documents]."""
    lens = np.asarray(seq_lens, dtype=np.int64)
    if lens.ndim == 1:
        lens = lens[None, :]
    out = np.zeros((lens.shape[0], seq_len), dtype=np.int32)
    for b in range(lens.shape[0]):
        cu = [0]
        for x in lens[b]:
            if x == padding_value:
                continue
            if x < 0:
                raise ValueError("a document length is negative")
            cu.append(cu[-1] + int(x))
        out[b] = doc_ids_from_cu_seqlens(cu, seq_len)
    return out


def position_ids_from_doc_ids(doc_ids):
    """(positions int32 [B, S], keep bool [B, S]) from document ids [B, S]."""
    ids = np.asarray(doc_ids)
    if ids.ndim == 1:
        ids = ids[None, :]
    B, S = ids.shape
    pos = np.zeros((B, S), dtype=np.int32)
    keep = ids != PAD_DOC_ID
    for b in range(B):
        start = 0
        for p in range(S):
            if p > 0 and ids[b, p] != ids[b, p - 1]:
                start = p
            if keep[b, p]:
                pos[b, p] = p - start
    return pos, keep


def validate_document_positions(keep, positions) -> np.ndarray:
    """First offending column of each row of (keep [B, S], positions [B, S]), or -1."""
    kp = np.asarray(keep).astype(bool)
    ps = np.asarray(positions).astype(np.int64)
    if kp.ndim == 1:
        kp, ps = kp[None, :], ps[None, :]
    bad = np.full(kp.shape[0], -1, dtype=np.int32)
    for b in range(kp.shape[0]):
        prev = -1
        for p in range(kp.shape[1]):
            if not kp[b, p]:
                continue
            x = ps[b, p]
            if prev < 0:
                ok = x >= 0
            elif prev == p - 1:
                ok = x == 0 or x == ps[b, prev] + 1
            else:
                ok = x == 0
            if not ok:
                bad[b] = p
                break
            prev = p
    return bad


def kv_needed_range(doc_ids_row, seq_start: int, L: int):
    """[lo, hi) of the key/value rows the local queries [seq_start, seq_start + L) attend."""
    ids = np.asarray(doc_ids_row).reshape(-1)
    lo, hi = None, None
    seg_start = 0
    for t in range(seq_start + L):
        if t > 0 and ids[t] != ids[t - 1]:
            seg_start = t
        if t >= seq_start and ids[t] != PAD_DOC_ID:
            lo = seg_start if lo is None else lo
            hi = t + 1
    if lo is None:
        return seq_start, seq_start
    return lo, hi


def kv_rows_per_shard(lo: int, hi: int, S: int, L: int) -> np.ndarray:
    """Rows of [lo, hi) in each shard [r L, min((r + 1) L, S)) of the row."""
    n = -(-S // L)
    out = np.zeros(n, dtype=np.int32)
    for j in range(lo, hi):
        out[j // L] += 1
    return out
