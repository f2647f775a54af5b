"""Tensor-level API over the C ABI: doc ids, segments, plan, and autograd attention.

Everything here allocates torch tensors and forwards pointers to
``libbd_attn.so`` through ``_native``; every computation runs in the
library's CUDA kernels.

Names follow the NeMo Automodel API reference pages:
``doc_ids_from_cu_seqlens`` / ``segment_cu_seqlens`` ("nemo_automodel
.components.models.glm5_next.cp") and ``cp_blockdiag_sdpa``
("nemo_automodel.components.distributed.blockdiag_cp").
"""
from __future__ import annotations

import torch

from . import _native as N

_status_words: dict[int, torch.Tensor] = {}


def device_status_word(device=None) -> torch.Tensor:
    """The per-device int32 status word the kernels report device-side errors into."""
    dev = torch.device(device if device is not None else "cuda")
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    w = _status_words.get(idx)
    if w is None:
        w = torch.zeros(1, dtype=torch.int32, device=torch.device("cuda", idx))
        _status_words[idx] = w
    return w


def check_device_status(device=None, reset: bool = True) -> None:
    """Synchronise and raise if a kernel reported an error since the last check."""
    w = device_status_word(device)
    code = N.bd_get_device_status(w)
    if reset:
        w.zero_()
    if code != N.BD_OK:
        exc = ValueError if code == N.BD_ERR_INVALID_ARG else RuntimeError
        raise exc(f"device reported: {N.status_string(code)} (status {code})")


def _csr(cu_seqlens, device):
    """(flat boundaries, row_ptr) int32 device tensors from one row or a list of rows."""
    if isinstance(cu_seqlens, (list, tuple)) and len(cu_seqlens) > 0 and (
            isinstance(cu_seqlens[0], torch.Tensor) or hasattr(cu_seqlens[0], "__len__")):
        rows = [torch.as_tensor(c, dtype=torch.int32).reshape(-1) for c in cu_seqlens]
    else:
        rows = [torch.as_tensor(cu_seqlens, dtype=torch.int32).reshape(-1)]
    lens = torch.tensor([0] + [r.numel() for r in rows], dtype=torch.int64).cumsum(0)
    flat = torch.cat([r.to("cpu") for r in rows]).to(device)
    return flat, lens.to(torch.int32).to(device), len(rows)


def doc_ids_from_cu_seqlens(cu_seqlens, seq_len: int, device=None, row_ptr=None) -> torch.Tensor:
    """Document ids [B, S] (int32, 0 == padding) from cumulative boundaries.

    ``cu_seqlens`` is one row's boundaries, a list of rows, or (with
    ``row_ptr``) the concatenated rows as a CUDA int32 tensor.
    """
    if row_ptr is not None:
        flat, rp, B = cu_seqlens, row_ptr, row_ptr.numel() - 1
    else:
        dev = device if device is not None else (
            cu_seqlens.device if isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda
            else "cuda")
        flat, rp, B = _csr(cu_seqlens, dev)
    ids = torch.empty((B, seq_len), dtype=torch.int32, device=flat.device)
    N.bd_doc_ids_from_cu_seqlens(flat, rp, B, seq_len, ids, device_status_word(flat.device))
    return ids


def segment_cu_seqlens(doc_ids: torch.Tensor):
    """(seg [B, S+1], seg_ids [B, S], nseg [B]) for ids [B, S] or [S]."""
    ids = doc_ids.reshape(-1, doc_ids.shape[-1]).to(torch.int32).contiguous()
    B, S = ids.shape
    seg = torch.empty((B, S + 1), dtype=torch.int32, device=ids.device)
    seg_ids = torch.empty((B, S), dtype=torch.int32, device=ids.device)
    nseg = torch.empty((B,), dtype=torch.int32, device=ids.device)
    N.bd_segment_cu_seqlens(ids, B, S, seg, seg_ids, nseg)
    return seg, seg_ids, nseg


def make_plan(seg, seg_ids, nseg, Hq: int, Hkv: int, L: int, seq_start: int = 0) -> torch.Tensor:
    """Plan buffer (uint8, device) for attention of L local queries against S keys."""
    B, S = seg_ids.shape
    plan = torch.empty(N.bd_attn_plan_size(B, Hq, Hkv, L, S), dtype=torch.uint8,
                       device=seg.device)
    N.bd_attn_plan(seg, seg_ids, nseg, B, Hq, Hkv, L, S, seq_start, plan)
    return plan


def _resolve_scale(scale, D):
    return float(D) ** -0.5 if scale is None else float(scale)


def attn_forward(q, k, v, plan, seq_start=0, scale=None, enable_gqa=False, keep_o16=True,
                 workspace=None, dropout_p: float = 0.0, seed: int = 0, offset: int = 0):
    """out [B,Hq,L,D] bf16, lse [B,Hq,L] fp32 and an fp16 copy of O (no autograd).

    The fp16 copy (same shape as out, without the dropout factor 1 / (1 - p);
    None when ``keep_o16`` is False) lets the backward form Delta = <dout, O>
    from O at 11 significant bits instead of out's 8.
    ``workspace`` (uint8, at least bd_attn_fwd_planned_workspace_size bytes) is
    allocated here when not given.  ``dropout_p`` > 0 drops attention weights
    with the counter-based mask of (seed, offset); the backward must be given
    the same three values.
    """
    B, Hq, L, D = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    if workspace is None:
        workspace = torch.empty(N.bd_attn_fwd_planned_workspace_size(B, Hkv, S, D),
                                dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q)
    out16 = torch.empty_like(q, dtype=torch.float16) if keep_o16 else None
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device)
    if dropout_p != 0.0:  # the library rejects p outside [0, 1)
        N.bd_attn_fwd_dropout_planned(q, k, v, B, Hq, Hkv, L, S, D, seq_start,
                                      _resolve_scale(scale, D), enable_gqa, plan, out, lse,
                                      dropout_p, seed, offset, out16, workspace,
                                      device_status_word(q.device))
    else:
        N.bd_attn_fwd_planned(q, k, v, B, Hq, Hkv, L, S, D, seq_start, _resolve_scale(scale, D),
                              enable_gqa, plan, out, lse, out16, workspace,
                              device_status_word(q.device))
    return out, lse, out16


def attn_backward(q, k, v, out, lse, dout, plan, seq_start=0, scale=None, enable_gqa=False,
                  workspace=None, out16=None, dropout_p: float = 0.0, seed: int = 0,
                  offset: int = 0):
    """dq, dk, dv (bf16) for the forward above (no autograd)."""
    B, Hq, L, D = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    if workspace is None:
        workspace = torch.empty(N.bd_attn_bwd_planned_workspace_size(B, Hq, Hkv, L, S, D),
                                dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    if dropout_p != 0.0:
        N.bd_attn_bwd_dropout_planned(q, k, v, out, lse, dout, B, Hq, Hkv, L, S, D, seq_start,
                                      _resolve_scale(scale, D), enable_gqa, plan, dq, dk, dv,
                                      workspace, dropout_p, seed, offset, out16,
                                      device_status_word(q.device))
    else:
        N.bd_attn_bwd_planned(q, k, v, out, lse, dout, B, Hq, Hkv, L, S, D, seq_start,
                              _resolve_scale(scale, D), enable_gqa, plan, dq, dk, dv, workspace,
                              out16, device_status_word(q.device))
    return dq, dk, dv


def cu_csr(cu_seqlens, device):
    """(flat boundaries, row_ptr) int32 device tensors for one row's boundaries or a list of
    rows, the layout bd_attn_fwd / bd_attn_bwd take."""
    flat, rp, _ = _csr(cu_seqlens, device)
    return flat, rp


def attn_forward_cu(q, k, v, cu_seqlens, row_ptr, seq_start=0, scale=None, enable_gqa=False,
                    workspace=None, dropout_p: float = 0.0, seed: int = 0, offset: int = 0):
    """out, lse and the workspace of the single-call forward (bd_attn_fwd, no autograd).

    ``cu_seqlens`` / ``row_ptr`` are the int32 device tensors of ``cu_csr``.  The
    workspace (bd_attn_workspace_size bytes, allocated here when not given)
    carries the plan and the fp16 copy of O to ``attn_backward_cu``.
    """
    B, Hq, L, D = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    if workspace is None:
        workspace = torch.empty(N.bd_attn_workspace_size(B, Hq, Hkv, L, S, D), dtype=torch.uint8,
                                device=q.device)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device)
    st = device_status_word(q.device)
    if dropout_p != 0.0:
        N.bd_attn_fwd_dropout(q, k, v, B, Hq, Hkv, L, S, D, cu_seqlens, row_ptr, seq_start,
                              _resolve_scale(scale, D), enable_gqa, out, lse, workspace,
                              dropout_p, seed, offset, st)
    else:
        N.bd_attn_fwd(q, k, v, B, Hq, Hkv, L, S, D, cu_seqlens, row_ptr, seq_start,
                      _resolve_scale(scale, D), enable_gqa, out, lse, workspace, st)
    return out, lse, workspace


def attn_backward_cu(q, k, v, out, lse, dout, cu_seqlens, row_ptr, workspace, seq_start=0,
                     scale=None, enable_gqa=False, dropout_p: float = 0.0, seed: int = 0,
                     offset: int = 0):
    """dq, dk, dv of the single-call backward (bd_attn_bwd, no autograd), on the
    workspace the forward used."""
    B, Hq, L, D = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    st = device_status_word(q.device)
    if dropout_p != 0.0:
        N.bd_attn_bwd_dropout(q, k, v, out, lse, dout, B, Hq, Hkv, L, S, D, cu_seqlens, row_ptr,
                              seq_start, _resolve_scale(scale, D), enable_gqa, dq, dk, dv,
                              workspace, dropout_p, seed, offset, st)
    else:
        N.bd_attn_bwd(q, k, v, out, lse, dout, B, Hq, Hkv, L, S, D, cu_seqlens, row_ptr,
                      seq_start, _resolve_scale(scale, D), enable_gqa, dq, dk, dv, workspace, st)
    return dq, dk, dv


class BlockdiagAttention(torch.autograd.Function):
    """Autograd wrapper: forward and backward both run the library's kernels."""

    @staticmethod
    def forward(ctx, q, k, v, plan, seq_start, scale, enable_gqa, dropout_p=0.0, seed=0,
                offset=0):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        out, lse, out16 = attn_forward(q, k, v, plan, seq_start, scale, enable_gqa,
                                        dropout_p=dropout_p, seed=seed, offset=offset)
        ctx.save_for_backward(q, k, v, out, lse, plan, out16)
        ctx.args = (seq_start, scale, enable_gqa, dropout_p, seed, offset)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, out, lse, plan, out16 = ctx.saved_tensors
        seq_start, scale, enable_gqa, dropout_p, seed, offset = ctx.args
        dq, dk, dv = attn_backward(q, k, v, out, lse, dout.contiguous(), plan, seq_start, scale,
                                   enable_gqa, out16=out16, dropout_p=dropout_p, seed=seed,
                                   offset=offset)
        return dq, dk, dv, None, None, None, None, None, None, None


def _draw_seed() -> int:
    """A 64-bit dropout seed from torch's default CPU generator (no device sync)."""
    return int(torch.randint(0, 2 ** 62, (1,), dtype=torch.int64).item())


def blockdiag_attention(q, k, v, *, cu_seqlens=None, doc_ids=None, seq_start: int = 0,
                        scale=None, enable_gqa: bool = False, return_lse: bool = False,
                        dropout_p: float = 0.0, dropout_seed=None, dropout_offset: int = 0):
    """Block-diagonal causal attention of q [B,Hq,L,D] against k, v [B,Hkv,S,D].

    The mask comes from ``doc_ids`` [B, S] (0 == padding) or, when those are
    not given, from ``cu_seqlens`` (one row's boundaries or a list of rows).
    ``dropout_p`` in [0, 1) drops attention weights with probability p',
    p rounded down to a multiple of 2^-16 (kept ones scaled by 1 / (1 - p'));
    the mask is a function of (dropout_seed, dropout_offset) and the
    positions, and the seed is drawn from torch's generator when None.
    """
    if not 0.0 <= float(dropout_p) < 1.0:
        raise ValueError("dropout_p must lie in [0, 1)")
    S = k.shape[2]
    if doc_ids is None:
        if cu_seqlens is None:
            raise ValueError("cu_seqlens or doc_ids is required")
        doc_ids = doc_ids_from_cu_seqlens(cu_seqlens, S, device=q.device)
    seg, seg_ids, nseg = segment_cu_seqlens(doc_ids)
    if seg_ids.shape[0] != q.shape[0]:
        raise ValueError("document ids must have one row per batch row")
    plan = make_plan(seg, seg_ids, nseg, q.shape[1], k.shape[1], q.shape[2], seq_start)
    seed = 0
    if dropout_p > 0.0:
        seed = _draw_seed() if dropout_seed is None else int(dropout_seed)
    out, lse = BlockdiagAttention.apply(q, k, v, plan, seq_start, scale, enable_gqa,
                                        float(dropout_p), seed, int(dropout_offset))
    return (out, lse) if return_lse else out


def cp_blockdiag_sdpa(query, key, value, attn_mask=None, dropout_p: float = 0.0,
                      is_causal: bool = False, scale=None, enable_gqa: bool = False, *,
                      doc_ids=None, cu_seqlens=None, seq_start: int = 0, dropout_seed=None,
                      dropout_offset: int = 0, **kwargs):
    """SDPA-shaped entry: local queries against delivered K/V, per-document causal mask.

    As on the page "nemo_automodel.components.distributed.blockdiag_cp",
    ``attn_mask`` and ``is_causal`` are ignored (the mask is rebuilt from the
    document ids), ``scale`` None means D**-0.5, and extra keyword arguments
    are accepted and ignored.  ``dropout_p`` acts as in torch's SDPA (on the
    normalised weights, applied whenever it is > 0), with p rounded down to a
    multiple of 2^-16 and kept weights scaled by 1 / (1 - p') for that p';
    ``dropout_seed`` / ``dropout_offset`` fix the mask (the seed is drawn
    from torch's generator when None).
    """
    del attn_mask, is_causal, kwargs
    return blockdiag_attention(query, key, value, cu_seqlens=cu_seqlens, doc_ids=doc_ids,
                               seq_start=seq_start, scale=scale, enable_gqa=enable_gqa,
                               dropout_p=dropout_p, dropout_seed=dropout_seed,
                               dropout_offset=dropout_offset)


def useful_pairs(cu_rows, seq_start: int, L: int) -> int:
    """Number of (query, key) pairs the mask allows, from host boundary lists (for FLOP counts)."""
    total = 0
    for cu in cu_rows:
        cu = [int(x) for x in cu]
        for a, b in zip(cu[:-1], cu[1:]):
            lo, hi = max(a, seq_start), min(b, seq_start + L)
            for_rows = 0
            if lo < hi:
                # rows t in [lo, hi) attend t - a + 1 keys each
                n1, n2 = lo - a + 1, hi - a
                for_rows = (n1 + n2) * (n2 - n1 + 1) // 2
            total += for_rows
    return total


__all__ = [
    "BlockdiagAttention", "attn_backward", "attn_backward_cu", "attn_forward", "attn_forward_cu",
    "blockdiag_attention", "cu_csr",
    "check_device_status", "cp_blockdiag_sdpa", "device_status_word", "doc_ids_from_cu_seqlens",
    "make_plan", "segment_cu_seqlens", "useful_pairs",
]
