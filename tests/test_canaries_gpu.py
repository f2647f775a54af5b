"""No entry point writes outside the buffers it was given.

Every output and workspace here sits inside a larger allocation with guard
regions of 4096 bytes on both sides, all filled with a sentinel byte before
the call.  After the calls (and a synchronisation) every guard byte must
still hold the sentinel.  The kernels mix TMA stores, which clip at a
tensor's extent, with plain stores from registers and shared memory, which do
not; these cases put the edges where a plain store could overrun: lengths not
a multiple of 128, query intervals, head dims 64 and 128, an odd GQA group,
padding rows, dropout, and the 8192-token benchmark workload.  The interior
starts full of sentinel bytes as well, so the results are also compared with
the oracle: an output element the kernels never wrote would show there.
"""
import zlib

import numpy as np
import pytest
import torch

from _gpu_common import assert_close, assert_lse, rand_bf16, to64
from oracle import blockdiag as orc
from packed_sequence_block_gb300 import _native as N
from packed_sequence_block_gb300 import attention as A
from packed_sequence_block_gb300.workloads import make_qkv_do, make_workload

pytestmark = pytest.mark.gpu

GUARD = 4096      # bytes on each side; a multiple of 256 keeps the interior aligned
SENTINEL = 0xA5


class Guarded:
    """Allocations with sentinel-filled guard regions around each interior tensor."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype, nbytes=None):
        n = nbytes if nbytes is not None else int(np.prod(shape)) * torch.empty(
            0, dtype=dtype).element_size()
        buf = torch.full((GUARD + n + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.bufs.append((buf, n))
        inner = buf[GUARD:GUARD + n]
        return inner if dtype == torch.uint8 and nbytes is not None else inner.view(dtype).view(shape)

    def check(self, tag):
        torch.cuda.synchronize()
        for i, (buf, n) in enumerate(self.bufs):
            lo, hi = buf[:GUARD], buf[GUARD + n:]
            assert torch.all(lo == SENTINEL), f"{tag}: buffer {i} written before its start"
            assert torch.all(hi == SENTINEL), f"{tag}: buffer {i} written past its end"


CASES = {
    # name: (cu rows, S, L, seq_start, Hq, Hkv, D)
    "tiny": ([[0, 37, 137, 138, 202, 256]], 256, 256, 0, 4, 2, 64),
    "g3_two_rows_ragged": ([[0, 17, 260, 517], [0, 400]], 517, 517, 0, 6, 2, 128),
    "interval_unaligned": ([[0, 150, 600, 1024]], 1024, 300, 200, 4, 1, 64),
    "last_query_only": ([[0, 200, 333]], 333, 1, 332, 4, 2, 128),
    "padding_row": ([[0, 90, 190], [0]], 190, 190, 0, 2, 1, 128),
}


def _inputs(name, B, S, L, Hq, Hkv, D):
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()) ^ 0xC0FFEE)
    q, do = rand_bf16((B, Hq, L, D), g), rand_bf16((B, Hq, L, D), g)
    k, v = rand_bf16((B, Hkv, S, D), g), rand_bf16((B, Hkv, S, D), g)
    return q, k, v, do


def _planned(G, q, k, v, do, ids_np, s0, drop):
    """ids -> segments -> plan -> forward -> backward -> no-workspace backward, all guarded."""
    B, Hq, L, D = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    gqa = Hq != Hkv
    st = A.device_status_word()
    ids = G((B, S), torch.int32)
    ids.copy_(torch.from_numpy(ids_np))
    seg, sid, nseg = G((B, S + 1), torch.int32), G((B, S), torch.int32), G((B,), torch.int32)
    N.bd_segment_cu_seqlens(ids, B, S, seg, sid, nseg)
    plan = G(None, torch.uint8, N.bd_attn_plan_size(B, Hq, Hkv, L, S))
    N.bd_attn_plan(seg, sid, nseg, B, Hq, Hkv, L, S, s0, plan)
    out, out16 = G((B, Hq, L, D), torch.bfloat16), G((B, Hq, L, D), torch.float16)
    lse = G((B, Hq, L), torch.float32)
    fws = G(None, torch.uint8, N.bd_attn_fwd_planned_workspace_size(B, Hkv, S, D))
    dq, dk, dv = (G((B, Hq, L, D), torch.bfloat16), G((B, Hkv, S, D), torch.bfloat16),
                  G((B, Hkv, S, D), torch.bfloat16))
    bws = G(None, torch.uint8, N.bd_attn_bwd_planned_workspace_size(B, Hq, Hkv, L, S, D))
    scale = D ** -0.5
    if drop is None:
        N.bd_attn_fwd_planned(q, k, v, B, Hq, Hkv, L, S, D, s0, scale, gqa, plan, out, lse, out16,
                              fws, st)
        N.bd_attn_bwd_planned(q, k, v, out, lse, do, B, Hq, Hkv, L, S, D, s0, scale, gqa, plan,
                              dq, dk, dv, bws, out16, st)
    else:
        N.bd_attn_fwd_dropout_planned(q, k, v, B, Hq, Hkv, L, S, D, s0, scale, gqa, plan, out,
                                      lse, *drop, out16, fws, st)
        N.bd_attn_bwd_dropout_planned(q, k, v, out, lse, do, B, Hq, Hkv, L, S, D, s0, scale, gqa,
                                      plan, dq, dk, dv, bws, *drop, out16, st)
    res = (out, lse, dq, dk, dv)
    if drop is None and N.bd_attn_bwd_planned_workspace_size(B, Hq, Hkv, L, S, D) <= \
            N.NOALLOC_SCRATCH_BYTES:
        dq2, dk2, dv2 = (G((B, Hq, L, D), torch.bfloat16), G((B, Hkv, S, D), torch.bfloat16),
                         G((B, Hkv, S, D), torch.bfloat16))
        N.bd_attn_bwd_noalloc(q, k, v, out, lse, do, B, Hq, Hkv, L, S, D, s0, scale, gqa, plan,
                              dq2, dk2, dv2, out16, st)
        res = res + (dq2, dk2, dv2)
    return res


def _single_call(G, q, k, v, do, cu_rows, s0, drop):
    B, Hq, L, D = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    gqa = Hq != Hkv
    st = A.device_status_word()
    cu, rp = A.cu_csr(cu_rows, "cuda")
    out, lse = G((B, Hq, L, D), torch.bfloat16), G((B, Hq, L), torch.float32)
    dq, dk, dv = (G((B, Hq, L, D), torch.bfloat16), G((B, Hkv, S, D), torch.bfloat16),
                  G((B, Hkv, S, D), torch.bfloat16))
    ws = G(None, torch.uint8, N.bd_attn_workspace_size(B, Hq, Hkv, L, S, D))
    scale = D ** -0.5
    if drop is None:
        N.bd_attn_fwd(q, k, v, B, Hq, Hkv, L, S, D, cu, rp, s0, scale, gqa, out, lse, ws, st)
        N.bd_attn_bwd(q, k, v, out, lse, do, B, Hq, Hkv, L, S, D, cu, rp, s0, scale, gqa, dq, dk,
                      dv, ws, st)
    else:
        N.bd_attn_fwd_dropout(q, k, v, B, Hq, Hkv, L, S, D, cu, rp, s0, scale, gqa, out, lse, ws,
                              *drop, st)
        N.bd_attn_bwd_dropout(q, k, v, out, lse, do, B, Hq, Hkv, L, S, D, cu, rp, s0, scale, gqa,
                              dq, dk, dv, ws, *drop, st)
    return out, lse, dq, dk, dv


def _check_values(tag, res, exp):
    assert_close(f"{tag} out", to64(res[0]), exp[0])
    assert_lse(f"{tag} lse", to64(res[1]), exp[1])
    for j in range(2, len(res)):
        assert_close(f"{tag} grad {j}", to64(res[j]), exp[2 + (j - 2) % 3])


def _oracle(q, k, v, do, ids, s0, drop):
    gqa = q.shape[1] != k.shape[1]
    kw = {} if drop is None else dict(dropout_p=drop[0], seed=drop[1], offset=drop[2])
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, gqa, **kw)
    return (eo, el) + orc.blockdiag_sdpa_backward(q, k, v, do, ids, s0, None, gqa, out=eo,
                                                  lse=el, **kw)


@pytest.mark.parametrize("drop", [None, (0.25, 0xDEC0DE, 1)], ids=["plain", "dropout"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_attention_entry_points_stay_inside_their_buffers(cuda_lib, name, drop):
    cu_rows, S, L, s0, Hq, Hkv, D = CASES[name]
    B = len(cu_rows)
    q, k, v, do = _inputs(name, B, S, L, Hq, Hkv, D)
    ids = np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in cu_rows])
    G = Guarded()
    planned = _planned(G, q, k, v, do, ids, s0, drop)
    single = _single_call(G, q, k, v, do, cu_rows, s0, drop)
    A.check_device_status()
    G.check(name)
    exp = _oracle(q, k, v, do, ids, s0, drop)
    _check_values(f"{name} planned", planned, exp)
    _check_values(f"{name} single call", single, exp)


def test_index_and_layout_entry_points_stay_inside_their_buffers(cuda_lib):
    st = A.device_status_word()
    rows = [[0, 37, 137, 138, 202, 256], [0, 5, 5, 100], [0]]
    B, S, L = 3, 300, 100
    G = Guarded()
    cu, rp = A.cu_csr(rows, "cuda")
    ids = G((B, S), torch.int32)
    N.bd_doc_ids_from_cu_seqlens(cu, rp, B, S, ids, st)
    lens = torch.tensor([[37, 100, 1, 64, 54], [5, 0, 95, -1000, -1000],
                         [-1000] * 5], dtype=torch.int32, device="cuda")
    ids2 = G((B, S), torch.int32)
    N.bd_doc_ids_from_seq_lens(lens, B, 5, S, -1000, ids2, st)
    seg, sid, nseg = G((B, S + 1), torch.int32), G((B, S), torch.int32), G((B,), torch.int32)
    N.bd_segment_cu_seqlens(ids, B, S, seg, sid, nseg)
    pos, keep = G((B, S), torch.int32), G((B, S), torch.uint8)
    N.bd_position_ids_from_doc_ids(ids, B, S, pos, keep)
    bad = G((B,), torch.int32)
    N.bd_validate_document_positions(keep, pos, B, S, bad, st)
    rng_, shards = G((B, 2), torch.int32), G((B, -(-S // L)), torch.int32)
    N.bd_kv_needed_range(seg, sid, nseg, B, S, L, 200, rng_, shards)
    A.check_device_status()
    G.check("index and layout")
    exp = np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in rows])
    assert np.array_equal(ids.cpu().numpy(), exp)
    assert np.array_equal(ids2.cpu().numpy(), exp)
    assert torch.all(bad == -1)


def test_benchmark_workload_stays_inside_its_buffers(cuda_lib):
    wl = make_workload("lognormal8k", 0)
    q, k, v, do = make_qkv_do(wl, device="cuda", generator_device="cuda")
    G = Guarded()
    res = _single_call(G, q, k, v, do, wl.cu, 0, None)
    A.check_device_status()
    G.check("lognormal8k")
    ids = np.stack([orc.doc_ids_from_cu_seqlens(c, wl.S) for c in wl.cu])
    _check_values("lognormal8k", res, _oracle(q, k, v, do, ids, 0, None))
