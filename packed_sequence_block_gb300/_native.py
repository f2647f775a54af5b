"""ctypes binding of libbd_attn.so: the C ABI entry points under the same names.

Each wrapper only marshals arguments: torch tensors become device pointers
(``data_ptr()``), the stream defaults to torch's current CUDA stream, and a
non-zero status becomes an exception (ValueError for argument errors,
RuntimeError otherwise).  All computation happens in the library's kernels;
there is no CPU fallback, and loading fails loudly when the library has not
been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbd_attn.so")

BD_OK = 0
BD_ERR_INVALID_ARG = 1
BD_ERR_UNSUPPORTED = 2
BD_ERR_CUDA = 3
BD_ERR_TIMEOUT = 4
BD_ERR_WORKSPACE = 5

_c_int, _c_size, _c_float, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
_c_double, _c_u64, _c_u32 = ctypes.c_double, ctypes.c_uint64, ctypes.c_uint32

# name -> (restype, argtypes); mirrors include/bd_attn.h
SIGNATURES = {
    "bd_status_string": (ctypes.c_char_p, [_c_int]),
    "bd_version": (_c_int, []),
    "bd_doc_ids_from_cu_seqlens": (_c_int, [_vp, _vp, _c_int, _c_int, _vp, _vp, _vp]),
    "bd_segment_cu_seqlens": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _vp, _vp]),
    "bd_doc_ids_from_seq_lens": (_c_int, [_vp] + [_c_int] * 4 + [_vp, _vp, _vp]),
    "bd_position_ids_from_doc_ids": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _vp]),
    "bd_validate_document_positions": (_c_int, [_vp, _vp, _c_int, _c_int, _vp, _vp, _vp]),
    "bd_kv_needed_range": (_c_int, [_vp, _vp, _vp] + [_c_int] * 4 + [_vp, _vp, _vp]),
    "bd_attn_plan_size": (_c_size, [_c_int] * 5),
    "bd_attn_plan": (_c_int, [_vp, _vp, _vp] + [_c_int] * 6 + [_vp, _c_size, _vp]),
    "bd_attn_workspace_size": (_c_size, [_c_int] * 6),
    "bd_attn_fwd": (_c_int, [_vp] * 3 + [_c_int] * 6 + [_vp, _vp, _c_int, _c_float, _c_int,
                                                        _vp, _vp, _vp, _c_size, _vp, _vp]),
    "bd_attn_bwd": (_c_int, [_vp] * 6 + [_c_int] * 6 + [_vp, _vp, _c_int, _c_float, _c_int,
                                                        _vp, _vp, _vp, _vp, _c_size, _vp, _vp]),
    "bd_attn_bwd_stages": (_c_int, [_vp] * 6 + [_c_int] * 6 + [
        _vp, _vp, _c_int, _c_float, _c_int, _vp, _vp, _vp, _vp, _c_size, _vp, _c_int, _vp]),
    "bd_attn_fwd_dropout": (_c_int, [_vp] * 3 + [_c_int] * 6 + [
        _vp, _vp, _c_int, _c_float, _c_int, _vp, _vp, _vp, _c_size, _c_double, _c_u64, _c_u32,
        _vp, _vp]),
    "bd_attn_bwd_dropout": (_c_int, [_vp] * 6 + [_c_int] * 6 + [
        _vp, _vp, _c_int, _c_float, _c_int, _vp, _vp, _vp, _vp, _c_size, _c_double, _c_u64,
        _c_u32, _vp, _vp]),
    "bd_attn_fwd_planned_workspace_size": (_c_size, [_c_int] * 4),
    "bd_attn_fwd_planned": (_c_int, [_vp, _vp, _vp] + [_c_int] * 7 + [
        _c_float, _c_int, _vp, _c_size, _vp, _vp, _vp, _vp, _c_size, _vp, _vp]),
    "bd_attn_fwd_dropout_planned": (_c_int, [_vp, _vp, _vp] + [_c_int] * 7 + [
        _c_float, _c_int, _vp, _c_size, _vp, _vp, _vp, _vp, _c_size, _c_double, _c_u64, _c_u32,
        _vp, _vp]),
    "bd_attn_bwd_planned_workspace_size": (_c_size, [_c_int] * 6),
    "bd_attn_bwd_planned": (_c_int, [_vp] * 7 + [_c_int] * 7 + [
        _c_float, _c_int, _vp, _c_size, _vp, _vp, _vp, _vp, _c_size, _vp, _vp]),
    "bd_attn_bwd_dropout_planned": (_c_int, [_vp] * 7 + [_c_int] * 7 + [
        _c_float, _c_int, _vp, _c_size, _vp, _vp, _vp, _vp, _c_size, _c_double, _c_u64, _c_u32,
        _vp, _vp]),
    "bd_attn_bwd_noalloc": (_c_int, [_vp] * 7 + [_c_int] * 7 + [_c_float, _c_int, _vp, _c_size,
                                                                 _vp, _vp, _vp, _vp, _vp]),
    "bd_test_arm_wait_timeout": (_c_int, [_c_int, ctypes.c_uint]),
    "bd_get_device_status": (_c_int, [_vp, _vp, _vp]),
}

# Size of the fixed scratch array bd_attn_bwd_noalloc uses (BD_NOALLOC_SCRATCH_BYTES in
# include/bd_attn.h; a CPU test keeps the two equal).
NOALLOC_SCRATCH_BYTES = 16 << 20

_lib = None


def lib():
    """Load (once) and return the ctypes handle of the built library."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -m packed_sequence_block_gb300.build` "
                "(the CUDA library is required: there is no CPU fallback)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(code: int) -> str:
    return lib().bd_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code == BD_OK:
        return
    msg = f"{what}: {status_string(code)} (status {code})"
    if code in (BD_ERR_INVALID_ARG, BD_ERR_UNSUPPORTED, BD_ERR_WORKSPACE):
        raise ValueError(msg)
    raise RuntimeError(msg)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _want(t, dtype, name):
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


# ------------------------------------------------------------------ entry points

def bd_version() -> int:
    return int(lib().bd_version())


def bd_doc_ids_from_cu_seqlens(cu, row_ptr, B: int, S: int, doc_ids, dev_status=None,
                               stream=None) -> None:
    for t, n in ((cu, "cu"), (row_ptr, "row_ptr"), (doc_ids, "doc_ids")):
        _want(t, torch.int32, n)
    _check(lib().bd_doc_ids_from_cu_seqlens(_ptr(cu), _ptr(row_ptr), B, S, _ptr(doc_ids),
                                            _ptr(dev_status), _stream(stream)),
           "bd_doc_ids_from_cu_seqlens")


def bd_segment_cu_seqlens(doc_ids, B: int, S: int, seg, seg_ids, nseg, stream=None) -> None:
    for t, n in ((doc_ids, "doc_ids"), (seg, "seg"), (seg_ids, "seg_ids"), (nseg, "nseg")):
        _want(t, torch.int32, n)
    _check(lib().bd_segment_cu_seqlens(_ptr(doc_ids), B, S, _ptr(seg), _ptr(seg_ids), _ptr(nseg),
                                       _stream(stream)), "bd_segment_cu_seqlens")


def bd_doc_ids_from_seq_lens(seq_lens, B: int, ndocs: int, S: int, padding_value: int, doc_ids,
                             dev_status=None, stream=None) -> None:
    for t, n in ((seq_lens, "seq_lens"), (doc_ids, "doc_ids")):
        _want(t, torch.int32, n)
    _check(lib().bd_doc_ids_from_seq_lens(_ptr(seq_lens), B, ndocs, S, int(padding_value),
                                          _ptr(doc_ids), _ptr(dev_status), _stream(stream)),
           "bd_doc_ids_from_seq_lens")


def bd_position_ids_from_doc_ids(doc_ids, B: int, S: int, positions, keep, stream=None) -> None:
    for t, n in ((doc_ids, "doc_ids"), (positions, "positions")):
        _want(t, torch.int32, n)
    if keep.dtype not in (torch.uint8, torch.bool):
        raise ValueError(f"keep must be uint8 or bool, got {keep.dtype}")
    _check(lib().bd_position_ids_from_doc_ids(_ptr(doc_ids), B, S, _ptr(positions), _ptr(keep),
                                              _stream(stream)), "bd_position_ids_from_doc_ids")


def bd_validate_document_positions(keep, positions, B: int, S: int, first_bad, dev_status=None,
                                   stream=None) -> None:
    if keep.dtype not in (torch.uint8, torch.bool):
        raise ValueError(f"keep must be uint8 or bool, got {keep.dtype}")
    for t, n in ((positions, "positions"), (first_bad, "first_bad")):
        _want(t, torch.int32, n)
    _check(lib().bd_validate_document_positions(_ptr(keep), _ptr(positions), B, S,
                                                _ptr(first_bad), _ptr(dev_status),
                                                _stream(stream)),
           "bd_validate_document_positions")


def bd_kv_needed_range(seg, seg_ids, nseg, B: int, S: int, L: int, seq_start: int, kv_range,
                       shard_rows=None, stream=None) -> None:
    for t, n in ((seg, "seg"), (seg_ids, "seg_ids"), (nseg, "nseg"), (kv_range, "range")):
        _want(t, torch.int32, n)
    if shard_rows is not None:
        _want(shard_rows, torch.int32, "shard_rows")
    _check(lib().bd_kv_needed_range(_ptr(seg), _ptr(seg_ids), _ptr(nseg), B, S, L, seq_start,
                                    _ptr(kv_range), _ptr(shard_rows), _stream(stream)),
           "bd_kv_needed_range")


def bd_attn_plan_size(B: int, Hq: int, Hkv: int, L: int, S: int) -> int:
    return int(lib().bd_attn_plan_size(B, Hq, Hkv, L, S))


def bd_attn_plan(seg, seg_ids, nseg, B: int, Hq: int, Hkv: int, L: int, S: int, seq_start: int,
                 plan, stream=None) -> None:
    _check(lib().bd_attn_plan(_ptr(seg), _ptr(seg_ids), _ptr(nseg), B, Hq, Hkv, L, S, seq_start,
                              _ptr(plan), _nbytes(plan), _stream(stream)),
           "bd_attn_plan")


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _want_all(pairs, dtype):
    for t, n in pairs:
        _want(t, dtype, n)


# ---- single-call forms: cumulative boundaries and one workspace

def bd_attn_workspace_size(B: int, Hq: int, Hkv: int, L: int, S: int, D: int) -> int:
    return int(lib().bd_attn_workspace_size(B, Hq, Hkv, L, S, D))


def bd_attn_fwd(q, k, v, B: int, Hq: int, Hkv: int, L: int, S: int, D: int, cu_seqlens, row_ptr,
                seq_start: int, scale: float, enable_gqa: bool, out, lse, workspace,
                dev_status=None, stream=None) -> None:
    _want_all(((q, "q"), (k, "k"), (v, "v"), (out, "out")), torch.bfloat16)
    _want_all(((cu_seqlens, "cu_seqlens"), (row_ptr, "row_ptr")), torch.int32)
    _want(lse, torch.float32, "lse")
    _check(lib().bd_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, L, S, D, _ptr(cu_seqlens),
                             _ptr(row_ptr), seq_start, float(scale), int(bool(enable_gqa)),
                             _ptr(out), _ptr(lse), _ptr(workspace), _nbytes(workspace),
                             _ptr(dev_status), _stream(stream)), "bd_attn_fwd")


def bd_attn_bwd(q, k, v, out, lse, dout, B: int, Hq: int, Hkv: int, L: int, S: int, D: int,
                cu_seqlens, row_ptr, seq_start: int, scale: float, enable_gqa: bool, dq, dk, dv,
                workspace, dev_status=None, stream=None) -> None:
    _want_all(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"),
               (dk, "dk"), (dv, "dv")), torch.bfloat16)
    _want_all(((cu_seqlens, "cu_seqlens"), (row_ptr, "row_ptr")), torch.int32)
    _want(lse, torch.float32, "lse")
    _check(lib().bd_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), B, Hq,
                             Hkv, L, S, D, _ptr(cu_seqlens), _ptr(row_ptr), seq_start,
                             float(scale), int(bool(enable_gqa)), _ptr(dq), _ptr(dk), _ptr(dv),
                             _ptr(workspace), _nbytes(workspace), _ptr(dev_status),
                             _stream(stream)), "bd_attn_bwd")


def bd_attn_bwd_stages(q, k, v, out, lse, dout, B: int, Hq: int, Hkv: int, L: int, S: int,
                       D: int, cu_seqlens, row_ptr, seq_start: int, scale: float,
                       enable_gqa: bool, dq, dk, dv, workspace, dev_status=None, stages: int = 7,
                       stream=None) -> None:
    _check(lib().bd_attn_bwd_stages(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                    B, Hq, Hkv, L, S, D, _ptr(cu_seqlens), _ptr(row_ptr),
                                    seq_start, float(scale), int(bool(enable_gqa)), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(workspace), _nbytes(workspace),
                                    _ptr(dev_status), int(stages), _stream(stream)),
           "bd_attn_bwd_stages")


def bd_attn_fwd_dropout(q, k, v, B: int, Hq: int, Hkv: int, L: int, S: int, D: int, cu_seqlens,
                        row_ptr, seq_start: int, scale: float, enable_gqa: bool, out, lse,
                        workspace, dropout_p: float, seed: int, offset: int = 0, dev_status=None,
                        stream=None) -> None:
    _want_all(((q, "q"), (k, "k"), (v, "v"), (out, "out")), torch.bfloat16)
    _want_all(((cu_seqlens, "cu_seqlens"), (row_ptr, "row_ptr")), torch.int32)
    _want(lse, torch.float32, "lse")
    _check(lib().bd_attn_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, L, S, D,
                                     _ptr(cu_seqlens), _ptr(row_ptr), seq_start, float(scale),
                                     int(bool(enable_gqa)), _ptr(out), _ptr(lse),
                                     _ptr(workspace), _nbytes(workspace), float(dropout_p),
                                     int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF,
                                     _ptr(dev_status), _stream(stream)), "bd_attn_fwd_dropout")


def bd_attn_bwd_dropout(q, k, v, out, lse, dout, B: int, Hq: int, Hkv: int, L: int, S: int,
                        D: int, cu_seqlens, row_ptr, seq_start: int, scale: float,
                        enable_gqa: bool, dq, dk, dv, workspace, dropout_p: float, seed: int,
                        offset: int = 0, dev_status=None, stream=None) -> None:
    _want_all(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"),
               (dk, "dk"), (dv, "dv")), torch.bfloat16)
    _want_all(((cu_seqlens, "cu_seqlens"), (row_ptr, "row_ptr")), torch.int32)
    _want(lse, torch.float32, "lse")
    _check(lib().bd_attn_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                     _ptr(dout), B, Hq, Hkv, L, S, D, _ptr(cu_seqlens),
                                     _ptr(row_ptr), seq_start, float(scale),
                                     int(bool(enable_gqa)), _ptr(dq), _ptr(dk), _ptr(dv),
                                     _ptr(workspace), _nbytes(workspace), float(dropout_p),
                                     int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF,
                                     _ptr(dev_status), _stream(stream)), "bd_attn_bwd_dropout")


# ---- planned forms: a plan from bd_attn_plan, separate workspaces

def bd_attn_fwd_planned_workspace_size(B: int, Hkv: int, S: int, D: int) -> int:
    return int(lib().bd_attn_fwd_planned_workspace_size(B, Hkv, S, D))


def bd_attn_fwd_planned(q, k, v, B: int, Hq: int, Hkv: int, L: int, S: int, D: int,
                        seq_start: int, scale: float, enable_gqa: bool, plan, out, lse,
                        out16=None, workspace=None, dev_status=None, stream=None) -> None:
    _want_all(((q, "q"), (k, "k"), (v, "v"), (out, "out")), torch.bfloat16)
    if out16 is not None:
        _want(out16, torch.float16, "out16")
    _want(lse, torch.float32, "lse")
    _check(lib().bd_attn_fwd_planned(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, L, S, D, seq_start,
                                     float(scale), int(bool(enable_gqa)), _ptr(plan),
                                     _nbytes(plan), _ptr(out), _ptr(lse), _ptr(out16),
                                     _ptr(workspace), _nbytes(workspace), _ptr(dev_status),
                                     _stream(stream)), "bd_attn_fwd_planned")


def bd_attn_fwd_dropout_planned(q, k, v, B: int, Hq: int, Hkv: int, L: int, S: int, D: int,
                                seq_start: int, scale: float, enable_gqa: bool, plan, out, lse,
                                dropout_p: float, seed: int, offset: int = 0, out16=None,
                                workspace=None, dev_status=None, stream=None) -> None:
    _want_all(((q, "q"), (k, "k"), (v, "v"), (out, "out")), torch.bfloat16)
    if out16 is not None:
        _want(out16, torch.float16, "out16")
    _want(lse, torch.float32, "lse")
    _check(lib().bd_attn_fwd_dropout_planned(
        _ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, L, S, D, seq_start, float(scale),
        int(bool(enable_gqa)), _ptr(plan), _nbytes(plan), _ptr(out), _ptr(lse), _ptr(out16),
        _ptr(workspace), _nbytes(workspace), float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF,
        int(offset) & 0xFFFFFFFF, _ptr(dev_status), _stream(stream)),
        "bd_attn_fwd_dropout_planned")


def bd_attn_bwd_planned_workspace_size(B: int, Hq: int, Hkv: int, L: int, S: int, D: int) -> int:
    return int(lib().bd_attn_bwd_planned_workspace_size(B, Hq, Hkv, L, S, D))


def bd_attn_bwd_planned(q, k, v, out, lse, dout, B: int, Hq: int, Hkv: int, L: int, S: int,
                        D: int, seq_start: int, scale: float, enable_gqa: bool, plan, dq, dk, dv,
                        workspace, out16=None, dev_status=None, stream=None) -> None:
    _want_all(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"),
               (dk, "dk"), (dv, "dv")), torch.bfloat16)
    _want(lse, torch.float32, "lse")
    if out16 is not None:
        _want(out16, torch.float16, "out16")
    _check(lib().bd_attn_bwd_planned(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(out16),
                                     _ptr(lse), _ptr(dout), B, Hq, Hkv, L, S, D, seq_start,
                                     float(scale), int(bool(enable_gqa)), _ptr(plan),
                                     _nbytes(plan), _ptr(dq), _ptr(dk), _ptr(dv),
                                     _ptr(workspace), _nbytes(workspace), _ptr(dev_status),
                                     _stream(stream)), "bd_attn_bwd_planned")


def bd_attn_bwd_dropout_planned(q, k, v, out, lse, dout, B: int, Hq: int, Hkv: int, L: int,
                                S: int, D: int, seq_start: int, scale: float, enable_gqa: bool,
                                plan, dq, dk, dv, workspace, dropout_p: float, seed: int,
                                offset: int = 0, out16=None, dev_status=None,
                                stream=None) -> None:
    _want_all(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"),
               (dk, "dk"), (dv, "dv")), torch.bfloat16)
    _want(lse, torch.float32, "lse")
    if out16 is not None:
        _want(out16, torch.float16, "out16")
    _check(lib().bd_attn_bwd_dropout_planned(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(out16), _ptr(lse), _ptr(dout), B, Hq, Hkv,
        L, S, D, seq_start, float(scale), int(bool(enable_gqa)), _ptr(plan), _nbytes(plan),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), _nbytes(workspace), float(dropout_p),
        int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF, _ptr(dev_status),
        _stream(stream)), "bd_attn_bwd_dropout_planned")


def bd_attn_bwd_noalloc(q, k, v, out, lse, dout, B: int, Hq: int, Hkv: int, L: int, S: int,
                        D: int, seq_start: int, scale: float, enable_gqa: bool, plan, dq, dk, dv,
                        out16=None, dev_status=None, stream=None) -> None:
    """bd_attn_bwd_planned without a workspace argument: the library's own fixed scratch is used.

    For callers that cannot allocate device memory.  Problems whose workspace
    exceeds NOALLOC_SCRATCH_BYTES raise ValueError; calls that overlap on the
    GPU race on the shared scratch.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout"), (dq, "dq"),
                 (dk, "dk"), (dv, "dv")):
        _want(t, torch.bfloat16, n)
    _want(lse, torch.float32, "lse")
    if out16 is not None:
        _want(out16, torch.float16, "out16")
    _check(lib().bd_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(out16),
                                     _ptr(lse), _ptr(dout), B, Hq, Hkv, L, S, D, seq_start,
                                     float(scale), int(bool(enable_gqa)), _ptr(plan),
                                     _nbytes(plan), _ptr(dq), _ptr(dk),
                                     _ptr(dv), _ptr(dev_status), _stream(stream)),
           "bd_attn_bwd_noalloc")


def bd_test_arm_wait_timeout(which: int, limit_us: int) -> None:
    """Make the next launch of the forward (1) or backward main (2) kernel from this
    thread withhold its first tile and give up its waits after limit_us (test hook)."""
    _check(lib().bd_test_arm_wait_timeout(int(which), int(limit_us)), "bd_test_arm_wait_timeout")


def bd_get_device_status(dev_status, stream=None) -> int:
    """Synchronise the stream and return the device status word."""
    host = ctypes.c_int32(0)
    _check(lib().bd_get_device_status(_ptr(dev_status), ctypes.addressof(host), _stream(stream)),
           "bd_get_device_status")
    return int(host.value)
