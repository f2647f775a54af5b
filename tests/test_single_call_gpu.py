"""GPU parity of the single-call entry points bd_attn_fwd / bd_attn_bwd.

These take the rows' cumulative document boundaries and one workspace, as
cp_blockdiag_sdpa (page "nemo_automodel.components.distributed.blockdiag_cp")
rebuilds the mask from the document ids of doc_ids_from_cu_seqlens (page
"nemo_automodel.components.models.glm5_next.cp").  Every case goes through the
C ABI and is compared element by element with the fp64 oracle (same bar as
the other parity tests), and with the planned entry points on the same inputs
(out, lse, dk, dv bit for bit: the same kernels run on the same plan).  Also
covered: the backward on a workspace that no longer records the forward (Delta
from out alone, still within the bar), invalid boundaries (all padding plus a
status), dropout, and the benchmark workload at full size.
"""
import zlib

import numpy as np
import pytest
import torch

from _gpu_common import assert_close, assert_lse, gpu_forward_backward, rand_bf16, to64
from oracle import blockdiag as orc
from packed_sequence_block_gb300 import _native as N
from packed_sequence_block_gb300 import attention as A
from packed_sequence_block_gb300.workloads import make_qkv_do, make_workload

pytestmark = pytest.mark.gpu

CASES = {
    # name: (cu rows, S, L, seq_start, Hq, Hkv, D)
    "tiny": ([[0, 37, 137, 138, 202, 256]], 256, 256, 0, 4, 2, 64),
    "g3_two_rows_ragged": ([[0, 17, 260, 517], [0, 400]], 517, 517, 0, 6, 2, 128),
    "interval_unaligned": ([[0, 150, 600, 1024]], 1024, 300, 200, 4, 1, 64),
    "interval_aligned_g4": ([[0, 700, 1300, 2048]], 2048, 256, 768, 8, 2, 128),
    "zero_length_and_empty_row": ([[0, 0, 5, 5, 200, 200, 333], [0]], 384, 384, 0, 4, 4, 128),
    "one_token_docs": ([list(range(0, 257))], 256, 256, 0, 2, 2, 64),
}


def _ids(cu_rows, S):
    return np.stack([orc.doc_ids_from_cu_seqlens(c, S) for c in cu_rows])


def _single_call(q, k, v, do, cu_rows, seq_start, dropout=None):
    p, seed, off = dropout if dropout is not None else (0.0, 0, 0)
    gqa = q.shape[1] != k.shape[1]
    cu, rp = A.cu_csr(cu_rows, q.device)
    out, lse, ws = A.attn_forward_cu(q, k, v, cu, rp, seq_start, None, gqa, dropout_p=p, seed=seed,
                                     offset=off)
    dq, dk, dv = A.attn_backward_cu(q, k, v, out, lse, do, cu, rp, ws, seq_start, None, gqa,
                                    dropout_p=p, seed=seed, offset=off)
    A.check_device_status(q.device)
    return out, lse, dq, dk, dv


def _inputs(name, B, S, L, Hq, Hkv, D):
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()))
    q, do = rand_bf16((B, Hq, L, D), g), rand_bf16((B, Hq, L, D), g)
    k, v = rand_bf16((B, Hkv, S, D), g), rand_bf16((B, Hkv, S, D), g)
    return q, k, v, do


@pytest.mark.parametrize("name", sorted(CASES))
def test_single_call_matches_oracle_and_planned(cuda_lib, name):
    cu_rows, S, L, s0, Hq, Hkv, D = CASES[name]
    B = len(cu_rows)
    q, k, v, do = _inputs(name, B, S, L, Hq, Hkv, D)
    got = _single_call(q, k, v, do, cu_rows, s0)
    ids = _ids(cu_rows, S)
    gqa = Hq != Hkv
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, gqa)
    edq, edk, edv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, s0, None, gqa, out=eo, lse=el)
    assert_close(f"{name} out", to64(got[0]), eo)
    assert_lse(f"{name} lse", to64(got[1]), el)
    assert_close(f"{name} dq", to64(got[2]), edq)
    assert_close(f"{name} dk", to64(got[3]), edk)
    assert_close(f"{name} dv", to64(got[4]), edv)
    planned = gpu_forward_backward(q, k, v, do, torch.from_numpy(ids).cuda(), s0)
    for i, label in ((0, "out"), (1, "lse"), (3, "dk"), (4, "dv")):
        assert torch.equal(got[i], planned[i]), f"{name}: {label} differs from the planned path"
    assert_close(f"{name} dq vs planned", to64(got[2]), to64(planned[2]))


def test_backward_without_the_forwards_record(cuda_lib):
    """A workspace that no longer records this out (another forward ran on it, or a
    fresh one) gives Delta from out alone: still within the bar."""
    cu_rows, S, L, s0, Hq, Hkv, D = CASES["g3_two_rows_ragged"]
    B = len(cu_rows)
    q, k, v, do = _inputs("record", B, S, L, Hq, Hkv, D)
    cu, rp = A.cu_csr(cu_rows, "cuda")
    out, lse, ws = A.attn_forward_cu(q, k, v, cu, rp, s0, None, True)
    A.attn_forward_cu(q, k, v, cu, rp, s0, None, True, workspace=ws)  # records another out
    ids = _ids(cu_rows, S)
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, s0, None, True)
    edq, edk, edv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, s0, None, True, out=eo, lse=el)
    for w in (ws, torch.zeros_like(ws)):
        dq, dk, dv = A.attn_backward_cu(q, k, v, out, lse, do, cu, rp, w, s0, None, True)
        A.check_device_status()
        assert_close("dq", to64(dq), edq)
        assert_close("dk", to64(dk), edk)
        assert_close("dv", to64(dv), edv)


def test_invalid_boundaries_are_padding_and_reported(cuda_lib):
    S, Hq, Hkv, D = 256, 2, 1, 64
    q, k, v, do = _inputs("invalid", 2, S, S, Hq, Hkv, D)
    rows = [[0, 100, 90, 256], [0, 128, 256]]  # row 0 decreases
    cu, rp = A.cu_csr(rows, "cuda")
    out, lse, ws = A.attn_forward_cu(q, k, v, cu, rp, 0, None, True)
    with pytest.raises(ValueError, match="invalid argument"):
        A.check_device_status()
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    eo, el = orc.blockdiag_sdpa_forward(q[1:], k[1:], v[1:], _ids([rows[1]], S), 0, None, True)
    assert_close("valid row out", to64(out[1:]), eo)


def test_single_call_dropout_matches_planned(cuda_lib):
    cu_rows, S, L, s0, Hq, Hkv, D = CASES["interval_unaligned"]
    q, k, v, do = _inputs("dropout", 1, S, L, Hq, Hkv, D)
    drop = (0.2, 0x5EED, 3)
    got = _single_call(q, k, v, do, cu_rows, s0, drop)
    planned = gpu_forward_backward(q, k, v, do, torch.from_numpy(_ids(cu_rows, S)).cuda(), s0,
                                   dropout=drop)
    for i, label in ((0, "out"), (1, "lse"), (3, "dk"), (4, "dv")):
        assert torch.equal(got[i], planned[i]), f"dropout: {label} differs from the planned path"
    assert_close("dropout dq vs planned", to64(got[2]), to64(planned[2]))


def test_single_call_lognormal8k_full(cuda_lib):
    wl = make_workload("lognormal8k", 0)
    q, k, v, do = make_qkv_do(wl, device="cuda", generator_device="cuda")
    got = _single_call(q, k, v, do, wl.cu, 0)
    ids = _ids(wl.cu, wl.S)
    eo, el = orc.blockdiag_sdpa_forward(q, k, v, ids, 0, None, True)
    edq, edk, edv = orc.blockdiag_sdpa_backward(q, k, v, do, ids, 0, None, True, out=eo, lse=el)
    assert_close("out", to64(got[0]), eo)
    assert_lse("lse", to64(got[1]), el)
    assert_close("dq", to64(got[2]), edq)
    assert_close("dk", to64(got[3]), edk)
    assert_close("dv", to64(got[4]), edv)


def test_workspace_size_covers_every_part(cuda_lib):
    B, Hq, Hkv, L, S, D = 1, 32, 8, 8192, 8192, 128
    one = N.bd_attn_workspace_size(B, Hq, Hkv, L, S, D)
    parts = (N.bd_attn_plan_size(B, Hq, Hkv, L, S)
             + N.bd_attn_fwd_planned_workspace_size(B, Hkv, S, D)
             + N.bd_attn_bwd_planned_workspace_size(B, Hq, Hkv, L, S, D) + 2 * B * Hq * L * D)
    assert one >= parts
