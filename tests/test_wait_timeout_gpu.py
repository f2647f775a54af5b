"""The bounded device-side waits: a wait that nothing completes gives up.

Every wait of the forward and backward kernels is bounded.  When one runs
out, the CTA records BD_ERR_TIMEOUT in the caller's status word, the other
roles of the CTA stop, each waits (bounded) for its own copies and
tensor-core work in flight, tensor memory is freed and the kernel returns.
The page "nemo_automodel.components.distributed.blockdiag_cp" asks the same
of its patch (attach_cp1_packed_varlen_hooks, always_call=True: a raising
forward must not leave anything behind); here it is the kernel that must not
hang or leave the device unusable.

bd_test_arm_wait_timeout makes the next launch withhold its producer's first
tile load (a barrier that nothing completes) and shortens the limit to 1 ms.
Each test checks that the call reports BD_ERR_TIMEOUT promptly, and then
runs the same problem normally on the same plan: its results must match the
oracle, which they only can if the timed-out launch left the plan's work
counters at zero and the device usable.
"""
import time
import zlib

import numpy as np
import pytest
import torch

from _gpu_common import assert_close, assert_lse, rand_bf16, to64
from oracle import blockdiag as orc
from packed_sequence_block_gb300 import _native as N
from packed_sequence_block_gb300 import attention as A

pytestmark = pytest.mark.gpu

LIMIT_US = 1000
CASES = {
    # name: (cu rows, S, Hq, Hkv, D)
    "tiny": ([[0, 37, 137, 138, 202, 256]], 256, 4, 2, 64),
    "g3_d128": ([[0, 17, 260, 517], [0, 400]], 517, 6, 2, 128),
}


def _inputs(name):
    cu_rows, S, Hq, Hkv, D = CASES[name]
    B = len(cu_rows)
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()))
    q, do = rand_bf16((B, Hq, S, D), g), rand_bf16((B, Hq, S, D), g)
    k, v = rand_bf16((B, Hkv, S, D), g), rand_bf16((B, Hkv, S, D), g)
    ids = np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in cu_rows])
    return q, k, v, do, ids


def _expect_timeout(fn):
    """Run fn (which launches work), then check the status word says the wait ran out."""
    t0 = time.perf_counter()
    fn()
    code = N.bd_get_device_status(A.device_status_word())
    elapsed = time.perf_counter() - t0
    A.device_status_word().zero_()
    assert code == N.BD_ERR_TIMEOUT, f"status {code}, expected BD_ERR_TIMEOUT"
    assert elapsed < 1.5, f"the timed-out launch took {elapsed:.2f} s"


def _oracle(q, k, v, do, ids):
    gqa = q.shape[1] != k.shape[1]
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, 0, None, gqa)
    return (eo, el) + orc.blockdiag_sdpa_backward(q, k, v, do, ids, 0, None, gqa, out=eo, lse=el)


def _compare(got, exp, tag):
    assert_close(f"{tag} out", to64(got[0]), exp[0])
    assert_lse(f"{tag} lse", to64(got[1]), exp[1])
    for i, name in ((2, "dq"), (3, "dk"), (4, "dv")):
        assert_close(f"{tag} {name}", to64(got[i]), exp[i])


@pytest.mark.parametrize("name", sorted(CASES))
def test_forward_wait_runs_out_then_the_plan_still_works(cuda_lib, name):
    q, k, v, do, ids = _inputs(name)
    gqa = q.shape[1] != k.shape[1]
    seg, sid, nseg = A.segment_cu_seqlens(torch.from_numpy(ids).cuda())
    plan = A.make_plan(seg, sid, nseg, q.shape[1], k.shape[1], q.shape[2], 0)
    A.check_device_status()
    N.bd_test_arm_wait_timeout(1, LIMIT_US)
    _expect_timeout(lambda: A.attn_forward(q, k, v, plan, 0, None, gqa))
    out, lse, out16 = A.attn_forward(q, k, v, plan, 0, None, gqa)
    dq, dk, dv = A.attn_backward(q, k, v, out, lse, do, plan, 0, None, gqa, out16=out16)
    A.check_device_status()
    _compare((out, lse, dq, dk, dv), _oracle(q, k, v, do, ids), f"{name} after forward timeout")


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_wait_runs_out_then_the_plan_still_works(cuda_lib, name):
    q, k, v, do, ids = _inputs(name)
    gqa = q.shape[1] != k.shape[1]
    seg, sid, nseg = A.segment_cu_seqlens(torch.from_numpy(ids).cuda())
    plan = A.make_plan(seg, sid, nseg, q.shape[1], k.shape[1], q.shape[2], 0)
    out, lse, out16 = A.attn_forward(q, k, v, plan, 0, None, gqa)
    A.check_device_status()
    N.bd_test_arm_wait_timeout(2, LIMIT_US)
    _expect_timeout(lambda: A.attn_backward(q, k, v, out, lse, do, plan, 0, None, gqa,
                                            out16=out16))
    dq, dk, dv = A.attn_backward(q, k, v, out, lse, do, plan, 0, None, gqa, out16=out16)
    A.check_device_status()
    _compare((out, lse, dq, dk, dv), _oracle(q, k, v, do, ids), f"{name} after backward timeout")


def test_single_call_forms_time_out_and_recover(cuda_lib):
    q, k, v, do, ids = _inputs("tiny")
    cu, rp = A.cu_csr(CASES["tiny"][0], "cuda")
    N.bd_test_arm_wait_timeout(1, LIMIT_US)
    _expect_timeout(lambda: A.attn_forward_cu(q, k, v, cu, rp, 0, None, True))
    out, lse, ws = A.attn_forward_cu(q, k, v, cu, rp, 0, None, True)
    A.check_device_status()
    N.bd_test_arm_wait_timeout(2, LIMIT_US)
    _expect_timeout(lambda: A.attn_backward_cu(q, k, v, out, lse, do, cu, rp, ws, 0, None, True))
    dq, dk, dv = A.attn_backward_cu(q, k, v, out, lse, do, cu, rp, ws, 0, None, True)
    A.check_device_status()
    _compare((out, lse, dq, dk, dv), _oracle(q, k, v, do, ids), "single call after timeouts")


def test_an_armed_request_is_used_once(cuda_lib):
    """The request covers one launch: the launch after it runs normally."""
    q, k, v, do, ids = _inputs("tiny")
    cu, rp = A.cu_csr(CASES["tiny"][0], "cuda")
    N.bd_test_arm_wait_timeout(1, LIMIT_US)
    _expect_timeout(lambda: A.attn_forward_cu(q, k, v, cu, rp, 0, None, True))
    for _ in range(2):
        out, lse, _ = A.attn_forward_cu(q, k, v, cu, rp, 0, None, True)
        A.check_device_status()
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, 0, None, True)
    assert_close("out", to64(out), eo)
    assert_lse("lse", to64(lse), el)
