"""Oracle: a plain fp64 CPU statement of block-diagonal causal attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import or run this module.  The product path (the
CUDA library and its Python binding) never imports it, and this module
imports nothing from the product package.

What it follows (NeMo Automodel API reference pages):

* "nemo_automodel.components.models.glm5_next.cp", functions
  ``doc_ids_from_cu_seqlens`` (cumulative boundaries -> ids [1, sequence]),
  ``segment_cu_seqlens`` (boundaries of runs of equal ids covering the whole
  row) and the data item ``_PAD_DOC_ID = 0``.
* "nemo_automodel.components.distributed.blockdiag_cp", function
  ``cp_blockdiag_sdpa``: local queries [B, Hq, L, D] attend the delivered keys
  [B, Hkv, S, D] under a per-document causal mask rebuilt from document ids,
  so packed documents never attend across a boundary; ``scale`` None means
  D**-0.5; ``enable_gqa`` as in torch SDPA.  ``enable_cp1_packed_varlen``
  fixes ``0 == padding`` for the ids.  ``Glm5NextPackedContext.seq_start``
  places the local rows at global positions ``seq_start + i``.

Readings where the pages are silent (each is listed in the design notes):

* documents are numbered 1..n in boundary order, a zero-length document
  still takes its number, positions past the last boundary get id 0;
* the mask of the query at global position t is the set of keys j <= t that
  lie in the same segment as t; a query in a padding segment (id 0) attends
  nothing, its output row is 0 and its log-sum-exp is -inf;
* the log-sum-exp is natural-log, scale included, one value per query row;
* query head h uses key/value head floor(h / (Hq / Hkv)).

The backward pass is the gradient of sum(out * dO) with respect to q, k, v,
written from the softmax derivative:  Delta_i = <dO_i, o_i>,
P_ij = exp(s_ij - lse_i), dS_ij = P_ij (<dO_i, v_j> - Delta_i),
dq_i = scale sum_j dS_ij k_j, dk_j = scale sum_i dS_ij q_i,
dv_j = sum_i P_ij dO_i (sums over the query heads sharing key head j).

Dropout (``dropout_p``, page "nemo_automodel.components.distributed.blockdiag_cp",
cp_blockdiag_sdpa) follows oracle/dropout.py.

Every segment is computed on its own with numpy fp64 matrix products; query
rows of one segment are processed in slices only to bound memory.
"""
from __future__ import annotations

import numpy as np

from .dropout import keep_mask, keep_scale

PAD_DOC_ID = 0

# query rows per slice when a segment's score block would be too large
_ROW_BUDGET = 1 << 24


def doc_ids_from_cu_seqlens(cu_seqlens, seq_len: int) -> np.ndarray:
    """Document id per position: d+1 on [cu[d], cu[d+1]), PAD_DOC_ID past cu[-1].

    Raises ValueError unless cu[0] == 0, cu is non-decreasing and cu[-1] <= seq_len.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64).reshape(-1)
    if cu.size < 1 or cu[0] != 0 or np.any(np.diff(cu) < 0) or cu[-1] > seq_len:
        raise ValueError("cu_seqlens must start at 0, be non-decreasing and end <= seq_len")
    ids = np.full(seq_len, PAD_DOC_ID, dtype=np.int32)
    for d in range(cu.size - 1):
        ids[cu[d]:cu[d + 1]] = d + 1
    return ids


def segment_cu_seqlens(doc_ids_row):
    """Boundaries of the maximal runs of equal ids, from 0 to len(row).

    Returns (seg, seg_ids): seg[k] is where run k starts (seg[-1] == len(row))
    and seg_ids[k] the id that run carries.  Padding runs are included.
    """
    ids = np.asarray(doc_ids_row).reshape(-1)
    S = ids.size
    starts = [0] + [p for p in range(1, S) if ids[p] != ids[p - 1]] if S > 0 else []
    seg = np.asarray(starts + [S], dtype=np.int32)
    seg_ids = np.asarray([ids[s] for s in starts], dtype=np.int32)
    return seg, seg_ids


def _segments(doc_ids_row):
    seg, seg_ids = segment_cu_seqlens(doc_ids_row)
    return [(int(seg[k]), int(seg[k + 1]), int(seg_ids[k])) for k in range(seg_ids.size)]


def _as_f64(x):
    if hasattr(x, "detach"):  # torch tensor (bf16 values are exact in fp64)
        import torch
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _check(q, k, v, seq_start, enable_gqa):
    B, Hq, L, D = q.shape
    Bk, Hkv, S, Dk = k.shape
    if v.shape != k.shape or Bk != B or Dk != D:
        raise ValueError("q [B,Hq,L,D], k and v [B,Hkv,S,D] required")
    if Hq % Hkv != 0 or (Hq != Hkv and not enable_gqa):
        raise ValueError("Hq must equal Hkv, or be a multiple of it with enable_gqa")
    if seq_start < 0 or seq_start + L > S:
        raise ValueError("need 0 <= seq_start and seq_start + L <= S")
    return B, Hq, Hkv, L, S, D


def _row_slices(t0, t1, n_keys):
    step = max(1, _ROW_BUDGET // max(1, n_keys))
    t = t0
    while t < t1:
        yield t, min(t1, t + step)
        t += step


def _mask_plane(mask_planes, b, h, Hq):
    return b * Hq + h if mask_planes is None else int(np.asarray(mask_planes)[b, h])


def blockdiag_sdpa_forward(q, k, v, doc_ids, seq_start=0, scale=None, enable_gqa=False,
                           dropout_p=0.0, seed=0, offset=0, mask_planes=None, mask_pos0=0):
    """out [B,Hq,L,D] and lse [B,Hq,L] in fp64 for block-diagonal causal attention.

    ``doc_ids`` is [B, S] (0 == padding).  Query i of q sits at global position
    seq_start + i and attends keys j <= seq_start + i of its own segment.
    With ``dropout_p`` > 0 the weights P are masked by oracle.dropout.keep_mask
    (``seed``, ``offset``) and kept ones scaled by oracle.dropout.keep_scale
    (1 / (1 - p') for p' = dropout_p rounded down to a multiple of 2^-16); lse is
    the softmax's, before dropout.  For a slice of a larger problem,
    ``mask_planes`` [B, Hq] gives each (row, head) its plane in the whole and
    ``mask_pos0`` the whole row's position of this row's position 0, so that
    the slice draws the whole problem's mask.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, Hq, Hkv, L, S, D = _check(q, k, v, seq_start, enable_gqa)
    ids = np.asarray(doc_ids).reshape(B, S)
    scale = D ** -0.5 if scale is None else float(scale)
    G = Hq // Hkv
    out = np.zeros((B, Hq, L, D))
    lse = np.full((B, Hq, L), -np.inf)
    for b in range(B):
        for start, end, sid in _segments(ids[b]):
            if sid == PAD_DOC_ID:
                continue
            t0, t1 = max(start, seq_start), min(end, seq_start + L)
            for r0, r1 in _row_slices(t0, t1, t1 - start):
                keys = np.arange(start, r1)
                allowed = keys[None, :] <= np.arange(r0, r1)[:, None]
                for h in range(Hq):
                    g = h // G
                    s = scale * (q[b, h, r0 - seq_start:r1 - seq_start] @ k[b, g, start:r1].T)
                    s = np.where(allowed, s, -np.inf)
                    m = s.max(axis=1, keepdims=True)
                    row_lse = m + np.log(np.exp(s - m).sum(axis=1, keepdims=True))
                    p = np.exp(s - row_lse)
                    if dropout_p > 0.0:
                        p = p * keep_mask(_mask_plane(mask_planes, b, h, Hq),
                                          np.arange(r0, r1) + mask_pos0, keys + mask_pos0,
                                          seed, offset, dropout_p) * keep_scale(dropout_p)
                    out[b, h, r0 - seq_start:r1 - seq_start] = p @ v[b, g, start:r1]
                    lse[b, h, r0 - seq_start:r1 - seq_start] = row_lse[:, 0]
    return out, lse


def blockdiag_sdpa_backward(q, k, v, dout, doc_ids, seq_start=0, scale=None,
                            enable_gqa=False, out=None, lse=None, dropout_p=0.0, seed=0,
                            offset=0, mask_planes=None, mask_pos0=0):
    """dq [B,Hq,L,D], dk and dv [B,Hkv,S,D] (fp64): gradient of sum(out * dout).

    ``out`` and ``lse`` default to this module's own forward pass.  dk/dv rows
    of keys no query of the interval attends are 0.  With dropout (mask M,
    r = keep_scale(p)): dv = (P o M r)^T dO and dS = P o (M r dP - Delta), where
    Delta = <dO, out> still equals sum_j P_ij M_ij r dP_ij.  ``mask_planes``
    and ``mask_pos0`` as in the forward.
    """
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, Hq, Hkv, L, S, D = _check(q, k, v, seq_start, enable_gqa)
    if out is None or lse is None:
        out, lse = blockdiag_sdpa_forward(q, k, v, doc_ids, seq_start, scale, enable_gqa,
                                          dropout_p, seed, offset, mask_planes, mask_pos0)
    ids = np.asarray(doc_ids).reshape(B, S)
    scale = D ** -0.5 if scale is None else float(scale)
    G = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    delta = (dout * out).sum(axis=-1)  # [B, Hq, L]
    for b in range(B):
        for start, end, sid in _segments(ids[b]):
            if sid == PAD_DOC_ID:
                continue
            t0, t1 = max(start, seq_start), min(end, seq_start + L)
            for r0, r1 in _row_slices(t0, t1, t1 - start):
                keys = np.arange(start, r1)
                allowed = keys[None, :] <= np.arange(r0, r1)[:, None]
                i0, i1 = r0 - seq_start, r1 - seq_start
                for h in range(Hq):
                    g = h // G
                    kk, vv = k[b, g, start:r1], v[b, g, start:r1]
                    s = scale * (q[b, h, i0:i1] @ kk.T)
                    p = np.where(allowed, np.exp(s - lse[b, h, i0:i1, None]), 0.0)
                    dp = dout[b, h, i0:i1] @ vv.T
                    pd = p
                    if dropout_p > 0.0:
                        mr = keep_mask(_mask_plane(mask_planes, b, h, Hq),
                                       np.arange(r0, r1) + mask_pos0, keys + mask_pos0, seed,
                                       offset, dropout_p) * keep_scale(dropout_p)
                        pd, dp = p * mr, dp * mr
                    ds = p * (dp - delta[b, h, i0:i1, None])
                    dq[b, h, i0:i1] = scale * (ds @ kk)
                    dk[b, g, start:r1] += scale * (ds.T @ q[b, h, i0:i1])
                    dv[b, g, start:r1] += pd.T @ dout[b, h, i0:i1]
    return dq, dk, dv
