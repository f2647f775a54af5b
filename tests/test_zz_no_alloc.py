"""The backward entry point for callers that cannot allocate device memory.

Some callers cannot hand the library a scratch buffer: code running inside a
host runtime that reserves all GPU memory when it starts and forbids later
allocations (an allocation can synchronise the device or fail once memory is
fragmented).  bd_attn_bwd_noalloc serves them with a fixed scratch array that
lives in the library image.  These tests call it through the C ABI, twice in a
row, and check each result against bd_attn_bwd (which takes a workspace) with
the tolerance the other parity tests use; they also check that a problem too
large for the fixed scratch is refused before anything runs.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from _gpu_common import assert_close, to64
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
    return q, k, v, do, plan


def test_noalloc_backward_matches_workspace_backward(cuda_lib):
    B, S, Hq, Hkv, D = 2, 700, 8, 2, 128
    q, k, v, do, plan = _problem(B, S, Hq, Hkv, D, [[0, 130, 400, 650], [0, 700]], 11)
    assert N.bd_attn_bwd_workspace_size(B, Hq, Hkv, S, S, D) <= N.NOALLOC_SCRATCH_BYTES
    out, lse, out_lo = A.attn_forward(q, k, v, plan, 0, None, True)
    ref = A.attn_backward(q, k, v, out, lse, do, plan, 0, None, True, out_lo=out_lo)
    A.check_device_status()
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        N.bd_attn_bwd_noalloc(q, k, v, out, lse, do, B, Hq, Hkv, S, S, D, 0, D ** -0.5, True,
                              plan, dq, dk, dv, out_lo=out_lo,
                              dev_status=A.device_status_word())
        A.check_device_status()
        assert_close(f"call {call} dq", to64(dq), to64(ref[0]))
        assert_close(f"call {call} dk", to64(dk), to64(ref[1]))
        assert_close(f"call {call} dv", to64(dv), to64(ref[2]))


def test_noalloc_refuses_problems_beyond_its_scratch(cuda_lib):
    B, S, Hq, Hkv, D = 1, 9000, 4, 4, 128
    assert N.bd_attn_bwd_workspace_size(B, Hq, Hkv, S, S, D) > N.NOALLOC_SCRATCH_BYTES
    q, k, v, do, plan = _problem(B, S, Hq, Hkv, D, [[0, 9000]], 12)
    out, lse = torch.empty_like(q), torch.zeros((B, Hq, S), device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    with pytest.raises(ValueError, match="too small"):
        N.bd_attn_bwd_noalloc(q, k, v, out, lse, do, B, Hq, Hkv, S, S, D, 0, D ** -0.5, False,
                              plan, dq, dk, dv, dev_status=A.device_status_word())
