"""The backward entry point for callers that cannot allocate device memory.

Some callers cannot hand the library a scratch buffer: code running inside a
host runtime that reserves all GPU memory when it starts and forbids later
allocations (an allocation can synchronise the device or fail once memory is
fragmented).  bd_attn_bwd_noalloc serves them with a fixed scratch array that
lives in the library image.  These tests call it through the C ABI, twice in a
row, and check each result against bd_attn_bwd_planned (which takes a
workspace): dk and dv bit for bit (they are deterministic), dq with the
tolerance the other parity tests use (its accumulation order varies).  A run
near the scratch limit is followed by a smaller problem of other shapes, so
that nothing an earlier, larger call left in the shared scratch can leak into
a later one; the smaller problem is also checked against the oracle.  A
problem too large for the fixed scratch is refused before anything runs.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from _gpu_common import assert_close, assert_lse, to64
from oracle import blockdiag as orc
from packed_sequence_block_gb300 import _native as N
from packed_sequence_block_gb300 import attention as A

pytestmark = pytest.mark.gpu


def _problem(B, S, Hq, Hkv, D, cu_rows, seed):
    g = torch.Generator().manual_seed(seed)
    rnd = lambda *s: torch.randn(s, generator=g).to(torch.bfloat16).cuda()  # noqa: E731
    q, do = rnd(B, Hq, S, D), rnd(B, Hq, S, D)
    k, v = rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    ids = np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in cu_rows])
    seg, sid, nseg = A.segment_cu_seqlens(torch.from_numpy(ids).cuda())
    plan = A.make_plan(seg, sid, nseg, Hq, Hkv, S, 0)
    return q, k, v, do, plan, ids


# (B, S, Hq, Hkv, D, cu rows, seed): the first needs 16,646,144 of the 16 MiB of
# scratch, the second has other L, Hq, G and D
NEAR_LIMIT = (1, 4000, 8, 2, 128, [[0, 1500, 3900]], 11)
SMALLER = (2, 700, 4, 1, 64, [[0, 130, 400, 650], [0, 700]], 12)


def _noalloc_against_workspace_path(case, calls=2):
    B, S, Hq, Hkv, D, cu_rows, seed = case
    q, k, v, do, plan, ids = _problem(B, S, Hq, Hkv, D, cu_rows, seed)
    gqa = Hq != Hkv
    assert N.bd_attn_bwd_planned_workspace_size(B, Hq, Hkv, S, S, D) <= N.NOALLOC_SCRATCH_BYTES
    out, lse, out16 = A.attn_forward(q, k, v, plan, 0, None, gqa)
    ref = A.attn_backward(q, k, v, out, lse, do, plan, 0, None, gqa, out16=out16)
    A.check_device_status()
    for call in range(calls):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        N.bd_attn_bwd_noalloc(q, k, v, out, lse, do, B, Hq, Hkv, S, S, D, 0, D ** -0.5, gqa,
                              plan, dq, dk, dv, out16=out16,
                              dev_status=A.device_status_word())
        A.check_device_status()
        assert_close(f"S={S} call {call} dq", to64(dq), to64(ref[0]))
        assert torch.equal(dk, ref[1]), f"S={S} call {call}: dk differs from the workspace path"
        assert torch.equal(dv, ref[2]), f"S={S} call {call}: dv differs from the workspace path"
    return q, k, v, do, ids, out, lse, (dq, dk, dv)


def test_noalloc_backward_matches_workspace_backward(cuda_lib):
    _noalloc_against_workspace_path(NEAR_LIMIT)
    q, k, v, do, ids, out, lse, (dq, dk, dv) = _noalloc_against_workspace_path(SMALLER)
    # and the smaller problem against the oracle
    gqa = q.shape[1] != k.shape[1]
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, 0, None, gqa)
    edq, edk, edv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, 0, None, gqa, out=eo, lse=el)
    assert_close("out", to64(out), eo)
    assert_lse("lse", to64(lse), el)
    assert_close("dq", to64(dq), edq)
    assert_close("dk", to64(dk), edk)
    assert_close("dv", to64(dv), edv)


def test_noalloc_refuses_problems_beyond_its_scratch(cuda_lib):
    B, S, Hq, Hkv, D = 1, 9000, 4, 4, 128
    assert N.bd_attn_bwd_planned_workspace_size(B, Hq, Hkv, S, S, D) > N.NOALLOC_SCRATCH_BYTES
    q, k, v, do, plan, _ = _problem(B, S, Hq, Hkv, D, [[0, 9000]], 12)
    out, lse = torch.empty_like(q), torch.zeros((B, Hq, S), device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    with pytest.raises(ValueError, match="too small"):
        N.bd_attn_bwd_noalloc(q, k, v, out, lse, do, B, Hq, Hkv, S, S, D, 0, D ** -0.5, False,
                              plan, dq, dk, dv, dev_status=A.device_status_word())
